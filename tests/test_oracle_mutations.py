"""The pins must catch plausible slips in the oracle.

Each case plants one mistake in the oracle (on the CPU, through monkeypatch),
runs the pin tests that guard that step, and expects at least one of them to
fail.  Nothing here touches the CUDA path.
"""

import math

import numpy as np
import pytest

from oracle import kvq_oracle as O
from tests import test_oracle_append as TA
from tests import test_oracle_attention as TT
from tests import test_oracle_quant as TQ
from tests import test_oracle_rotation as TR
from tests import test_oracle_size_law as TS


def _fails(fn, *args):
    try:
        fn(*args)
    except Exception:
        return True
    return False


def _quantize_floor(x, bits):
    x = np.asarray(x, np.float32)
    qmax = np.float32(O.QMAX[bits])
    s16 = np.minimum(np.max(np.abs(x), -1) / qmax, np.float32(65504)).astype(np.float16)
    sf = s16.astype(np.float32)[..., None]
    with np.errstate(all="ignore"):
        r = np.floor(x / sf + np.float32(0.5))  # round-half-up instead of half-to-even
    r = np.where(sf == 0, 0, r)
    return s16, np.clip(r, -qmax, qmax).astype(np.int8)


def _quantize_wrong_qmax(x, bits):
    x = np.asarray(x, np.float32)
    qmax = np.float32(2 ** (bits - 1))  # 8 instead of 7 for 4-bit
    s16 = np.minimum(np.max(np.abs(x), -1) / qmax, np.float32(65504)).astype(np.float16)
    sf = s16.astype(np.float32)[..., None]
    with np.errstate(all="ignore"):
        r = np.rint(x / sf)
    r = np.where(sf == 0, 0, r)
    return s16, np.clip(r, -qmax, qmax - 1).astype(np.int8)


def _pack_swapped(codes, bits):
    c = np.asarray(codes, np.int64)
    if bits == 4:
        u = (c + 8).reshape(*c.shape[:-1], c.shape[-1] // 2, 2)
        return (u[..., 1] | (u[..., 0] << 4)).astype(np.uint8)
    return _ORIG_PACK(codes, bits)


def _pack_3bit_bytewise(codes, bits):
    """A 3-bit packer that drops bits crossing a byte boundary."""
    c = np.asarray(codes, np.int64)
    if bits != 3:
        return _ORIG_PACK(codes, bits)
    u = (c + 4).reshape(*c.shape[:-1], c.shape[-1] // 8, 8)
    out = np.zeros((*u.shape[:-1], 3), np.int64)
    for j in range(8):
        pos = 3 * j
        out[..., pos // 8] |= (u[..., j] << (pos % 8)) & 0xFF
    return out.reshape(*c.shape[:-1], -1).astype(np.uint8)


def _fwht_missing_stage(x):
    y = np.asarray(x, np.float32)
    lead = y.shape[:-1]
    h = 1
    while h < 64:  # drops the stride-64 stage
        y = y.reshape(*lead, 128 // (2 * h), 2, h)
        a, b = y[..., 0, :], y[..., 1, :]
        y = np.stack([a + b, a - b], axis=-2).reshape(*lead, 128)
        h *= 2
    return y


def _attention_no_sqrt(q, K, V):
    q = np.asarray(q, np.float64)
    if K.shape[0] == 0:
        return np.zeros(q.shape[-1])
    s = np.asarray(K, np.float64) @ q
    return O.softmax_f64(s) @ np.asarray(V, np.float64)


def _scores_no_sqrt(q, K):
    return np.asarray(K, np.float64) @ np.asarray(q, np.float64)


def _rope_wrong_pairs(k, positions, theta):
    """Interleaved pairs (2i, 2i+1) instead of split halves."""
    k = np.asarray(k, np.float64)
    D = k.shape[-1]
    inv = theta ** (-2.0 * np.arange(D // 2) / D)
    ang = np.asarray(positions, np.float64).reshape(-1, *([1] * (k.ndim - 1))) * inv
    a, b = k[..., 0::2], k[..., 1::2]
    out = np.empty_like(k)
    out[..., 0::2] = a * np.cos(ang) - b * np.sin(ang)
    out[..., 1::2] = a * np.sin(ang) + b * np.cos(ang)
    return out


def _q_end_off_by_one(cfg, T):
    gam = O.unit_tokens(cfg)
    R = cfg.residual_window
    if T <= R:
        return 0
    return ((T - R + 1) // gam) * gam


def _block_bytes_no_scale(bits, group):
    return group * bits // 8 if bits != 16 else 2 * group


_ORIG_PACK = O.pack

MUTATIONS = {
    "round_half_up": ("quantize", _quantize_floor,
                      [(TQ.test_codes_are_nearest_grid_point, 4), (TQ.test_codes_are_nearest_grid_point, 2)]),
    "qmax_power_of_two": ("quantize", _quantize_wrong_qmax,
                          [(TQ.test_scale_follows_two_step_rounding, 4), (TQ.test_error_bound_half_scale, 4)]),
    "nibbles_swapped": ("pack", _pack_swapped, [(TQ.test_pack_every_code_at_every_position, 4, 32)]),
    "3bit_bytes_cut": ("pack", _pack_3bit_bytewise, [(TQ.test_three_bit_positions_three_to_seven_survive,)]),
    "fwht_stage_dropped": ("fwht_f32", _fwht_missing_stage,
                           [(TR.test_butterfly_equals_matrix_on_integers,)]),
    "attention_no_sqrt": ("attention_f64", _attention_no_sqrt, [(TT.test_two_tokens_closed_form_with_sqrt_d,)]),
    "scores_no_sqrt": ("scores_f64", _scores_no_sqrt, [(TT.test_key_error_identity,),
                                                       (TT.test_two_tokens_closed_form_with_sqrt_d,)]),
    "rope_interleaved": ("rope_f64", _rope_wrong_pairs, [(TT.test_rope_is_complex_rotation_of_split_halves,)]),
    "window_off_by_one": ("q_end", _q_end_off_by_one, [(TA.test_tier_boundaries_move_by_whole_groups,)]),
    "scale_bytes_dropped": ("block_bytes", _block_bytes_no_scale, [(TS.test_block_bytes_match_named_layouts,)]),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, monkeypatch, golden_dir):
    attr, fake, checks = MUTATIONS[name]
    # the unmutated pins pass
    for fn, *args in checks:
        assert not _fails(fn, *args), (name, fn.__name__)
    monkeypatch.setattr(O, attr, fake)
    assert any(_fails(fn, *args) for fn, *args in checks), name
