"""Pins of the oracle's append state machine: window, tiers, requantization,
paging.  Bulk append must leave the same live state as appending one token at
a time, and every dequantized value must sit within the quantizer's bound of
the input it came from."""

import numpy as np
import pytest

from oracle import kvq_oracle as O

KIVI = dict(k_fmt=O.Fmt(4, 32, O.AXIS_CHANNEL), v_fmt=O.Fmt(4, 32))
TIERS = dict(k_fmt=O.Fmt(4, 32, O.AXIS_CHANNEL), v_fmt=O.Fmt(4, 32),
             k_cold=O.Fmt(2, 32, O.AXIS_CHANNEL), v_cold=O.Fmt(2, 32))


def _inputs(cfg, n, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    k = (rng.standard_normal((n, cfg.H_kv, cfg.D)) * scale).astype(np.float16).view(np.uint16)
    v = (rng.standard_normal((n, cfg.H_kv, cfg.D)) * scale).astype(np.float16).view(np.uint16)
    return k, v


def _live_state(cfg, bufs, T, block_table=None):
    """Everything a decode step can read, per (layer, seq): dequantized K/V."""
    out = []
    for layer in range(cfg.L):
        for b in range(cfg.batch):
            out.append(O.dequantize(cfg, bufs, layer, b, int(T[b]), block_table=block_table))
    return out


CASES = {
    "per_token_q8_q4": O.Config(L=1, H_kv=2, H_q=2, D=128, batch=2, max_T=160,
                                k_fmt=O.Fmt(8, 32), v_fmt=O.Fmt(4, 32)),
    "per_token_window": O.Config(L=1, H_kv=2, H_q=4, D=128, batch=1, max_T=160,
                                 k_fmt=O.Fmt(4, 32), v_fmt=O.Fmt(4, 32), residual_window=20),
    "kivi_window": O.Config(L=2, H_kv=2, H_q=2, D=128, batch=2, max_T=200, residual_window=16, **KIVI),
    "kivi_no_window": O.Config(L=1, H_kv=1, H_q=1, D=128, batch=1, max_T=200, **KIVI),
    "rotated_3bit": O.Config(L=1, H_kv=2, H_q=4, D=256, batch=1, max_T=100,
                             k_fmt=O.Fmt(4, 128), v_fmt=O.Fmt(3, 128), flags=O.ROTATE_K | O.ROTATE_V,
                             sign_seed=3),
    "tiers": O.Config(L=1, H_kv=2, H_q=4, D=128, batch=2, max_T=400, hot_window=64,
                      residual_window=16, flags=O.K_PRE_ROPE, **TIERS),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_bulk_equals_token_by_token(name):
    cfg = CASES[name]
    T = {"per_token_q8_q4": [150, 97], "per_token_window": [130], "kivi_window": [190, 75],
         "kivi_no_window": [170], "rotated_3bit": [90], "tiers": [371, 200]}[name]
    total = sum(T)
    k, v = _inputs(cfg, total * cfg.L, 1)
    bulk = O.new_buffers(cfg)
    step = O.new_buffers(cfg)
    offs = np.concatenate([[0], np.cumsum(T)])
    for layer in range(cfg.L):
        kl, vl = k[layer * total:(layer + 1) * total], v[layer * total:(layer + 1) * total]
        O.append(cfg, bulk, layer, kl, vl, T, [0] * cfg.batch)
        # the same tokens in uneven chunks: 1, 3, 1, 7, 1, ...
        done = [0] * cfg.batch
        sizes = [1, 3, 1, 7, 1, 40, 1, 1, 33]
        i = 0
        while any(d < t for d, t in zip(done, T)):
            chunk = sizes[i % len(sizes)]
            i += 1
            n = [min(chunk, t - d) for d, t in zip(done, T)]
            ks = np.concatenate([kl[offs[b] + done[b]:offs[b] + done[b] + n[b]] for b in range(cfg.batch)])
            vs = np.concatenate([vl[offs[b] + done[b]:offs[b] + done[b] + n[b]] for b in range(cfg.batch)])
            O.append(cfg, step, layer, ks, vs, n, done)
            done = [d + x for d, x in zip(done, n)]
    for (kb, vb), (ks, vs) in zip(_live_state(cfg, bulk, T), _live_state(cfg, step, T)):
        assert np.array_equal(kb, ks) and np.array_equal(vb, vs)


def test_tier_boundaries_move_by_whole_groups():
    cfg = CASES["tiers"]
    for T in range(0, 400):
        qe, ce = O.q_end(cfg, T), O.c_end(cfg, T)
        assert qe % 32 == 0 and ce % 32 == 0 and 0 <= ce <= qe <= T
        if T >= 16:
            assert 16 <= T - qe < 16 + 32
        else:
            assert qe == 0
        if qe >= 64:
            assert 64 <= qe - ce < 64 + 32


def test_values_within_quantizer_bounds():
    cfg = CASES["kivi_window"]
    T = [190, 75]
    k, v = _inputs(cfg, sum(T) * cfg.L, 2)
    bufs = O.new_buffers(cfg)
    O.append(cfg, bufs, 0, k[:sum(T)], v[:sum(T)], T, [0, 0])
    K, V = O.dequantize(cfg, bufs, 0, 0, 190)
    kin = O.f16_bits_to_f32(k[:190]).astype(np.float64)
    vin = O.f16_bits_to_f32(v[:190]).astype(np.float64)
    qe = O.q_end(cfg, 190)
    assert qe == 160
    # window tokens are exact
    assert np.array_equal(K[qe:], kin[qe:]) and np.array_equal(V[qe:], vin[qe:])
    # per-channel K: error <= (scale/2)(1+2^-10) with scale ~ amax over 32 tokens / 7
    ka = np.abs(kin[:qe]).reshape(5, 32, 2, 128).max(axis=1)
    kerr = np.abs(K[:qe] - kin[:qe]).reshape(5, 32, 2, 128).max(axis=1)
    assert np.all(kerr <= ka / 7 * (1 + 2 ** -10) / 2 + ka * 2 ** -11)
    va = np.abs(vin[:qe]).reshape(qe, 2, 4, 32).max(axis=-1)
    verr = np.abs(V[:qe] - vin[:qe]).reshape(qe, 2, 4, 32).max(axis=-1)
    assert np.all(verr <= va / 7 * (1 + 2 ** -10) / 2 + va * 2 ** -11)


def test_cold_tier_is_requantized_from_hot_values():
    cfg = CASES["tiers"]
    T = [371, 200]
    k, v = _inputs(cfg, sum(T), 3)
    bufs = O.new_buffers(cfg)
    O.append(cfg, bufs, 0, k, v, T, [0, 0])
    ce = O.c_end(cfg, 371)
    assert ce == 288
    # rebuild group 0 of K by hand: 4-bit per channel, dequantize, 2-bit per channel
    x = O.f16_bits_to_f32(k[:32])  # [32, H, D]
    s4, c4 = O.quantize(np.transpose(x, (1, 2, 0)), 4)
    hot = O.dequantize_f32(s4, c4)
    s2, c2 = O.quantize(hot, 2)
    Kd, _ = O.dequantize(cfg, bufs, 0, 0, 371, 0, 32)
    assert np.array_equal(Kd, np.transpose(O.dequantize_f64(s2, c2), (2, 0, 1)))
    # 2-bit codes are ternary
    assert set(np.unique(c2)) <= {-1, 0, 1}


def test_paged_equals_contiguous():
    base = dict(L=2, H_kv=2, H_q=4, D=128, batch=3, max_T=96, k_fmt=O.Fmt(4, 128), v_fmt=O.Fmt(4, 128),
                flags=O.ROTATE_K | O.ROTATE_V, sign_seed=9)
    cont = O.Config(**base)
    paged = O.Config(**base, page_tokens=16, n_pages=20, max_pages_per_seq=6)
    rng = np.random.default_rng(4)
    table = rng.permutation(20)[:18].reshape(3, 6)
    T = [96, 33, 70]
    k, v = _inputs(cont, sum(T), 5)
    bc, bp = O.new_buffers(cont), O.new_buffers(paged)
    for layer in range(2):
        O.append(cont, bc, layer, k, v, T, [0, 0, 0])
        O.append(paged, bp, layer, k, v, T, [0, 0, 0], block_table=table)
    for layer in range(2):
        for b in range(3):
            a = O.dequantize(cont, bc, layer, b, T[b])
            p = O.dequantize(paged, bp, layer, b, T[b], block_table=table)
            assert np.array_equal(a[0], p[0]) and np.array_equal(a[1], p[1])


def test_window_covering_everything_is_plain_attention():
    cfg = O.Config(L=1, H_kv=1, H_q=2, D=128, batch=1, max_T=64, residual_window=64, **KIVI)
    k, v = _inputs(cfg, 50, 6)
    bufs = O.new_buffers(cfg)
    O.append(cfg, bufs, 0, k, v, [50], [0])
    assert O.q_end(cfg, 50) == 0
    q = np.random.default_rng(7).standard_normal((1, 1, 2, 128)).astype(np.float16).view(np.uint16)
    out = O.decode_attention(cfg, bufs, 0, 1, q, [50])
    K = O.f16_bits_to_f32(k)[:, 0].astype(np.float64)
    V = O.f16_bits_to_f32(v)[:, 0].astype(np.float64)
    for h in range(2):
        assert np.array_equal(out[0, 0, h], O.attention_f64(O.f16_bits_to_f32(q[0, 0, h]), K, V))


def test_hot_window_longer_than_cache_is_single_tier():
    cfg = CASES["tiers"]
    assert O.c_end(cfg, 64 + 16 + 31) == 0
    single = O.Config(**{**cfg.__dict__, "hot_window": 0, "k_cold": None, "v_cold": None})
    T = [100, 60]
    k, v = _inputs(cfg, sum(T), 8)
    a, b = O.new_buffers(cfg), O.new_buffers(single)
    O.append(cfg, a, 0, k, v, T, [0, 0])
    O.append(single, b, 0, k, v, T, [0, 0])
    for s in range(2):
        x, y = O.dequantize(cfg, a, 0, s, T[s]), O.dequantize(single, b, 0, s, T[s])
        assert np.array_equal(x[0], y[0]) and np.array_equal(x[1], y[1])


def test_capacity_is_enforced():
    cfg = CASES["per_token_q8_q4"]
    k, v = _inputs(cfg, 2, 9)
    with pytest.raises(ValueError):
        O.append(cfg, O.new_buffers(cfg), 0, k, v, [1, 1], [160, 0])
