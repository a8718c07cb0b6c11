"""The C-ABI library loads without a GPU, exports every symbol kvq.h declares,
and its host-side arithmetic (size law, buffer sizes, validation) agrees with
the oracle.  No kernel is launched here."""

import os
import re
import subprocess

import pytest

from oracle import kvq_oracle as O
from tests.helpers import oracle_cfg

K = pytest.importorskip("bit_kv_cache_04_gb300.kvq")
from bit_kv_cache_04_gb300 import workloads as W  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "kvq.h")).read()
    return sorted(set(re.findall(r"KVQ_API\s+[\w\s\*]+?\b(kvq_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    declared = _declared()
    assert len(declared) >= 16
    out = subprocess.run(["nm", "-D", "--defined-only", K.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (kvq_\w+)", out))
    assert set(declared) <= exported, set(declared) - exported
    assert set(K.EXPORTED) == set(declared)
    # nothing but the ABI is exported from the library's own code
    assert {s for s in exported if s.startswith("kvq")} == set(declared)


def test_version():
    assert "sm_103a" in K.kvq_version()


@pytest.mark.parametrize("bits,group,bb", [(8, 32, 34), (4, 32, 18), (4, 128, 66), (3, 128, 50), (2, 32, 10),
                                           (16, 128, 256)])
def test_block_bytes(bits, group, bb):
    assert K.kvq_block_bytes(bits, group) == bb == O.block_bytes(bits, group)


@pytest.mark.parametrize("name", W.ALL)
def test_size_law_matches_oracle(name):
    w = W.make(name, extra_tokens=0)
    oc = oracle_cfg(w.cfg)
    assert K.kvq_bytes_per_token(w.cfg) == O.bytes_per_token(oc)
    for T in (0, 1, 31, 32, 127, 128, 129, 160, 1000, 4096 + 160, w.cfg.max_T):
        assert K.kvq_cache_bytes(w.cfg, T) == O.cache_bytes(oc, T), T


def test_cache_identity_262k():
    # trefon.com, "Przyklad: model 27B przy 262K": 4224 MiB at 262,144 tokens (66 B/128)
    assert K.kvq_cache_bytes(W.make("ctx262k_hadamard4", 0).cfg, 262144) == 4224 * 2 ** 20
    assert K.kvq_cache_bytes(W.make("ctx262k_hadamard3", 0).cfg, 262144) == 3200 * 2 ** 20


@pytest.mark.parametrize("name", W.ALL)
def test_buffer_sizes_match_oracle_layout(name):
    w = W.make(name).scaled(L=2, lengths=[300, 77][: 1 if W.make(name).cfg.batch == 1 else 2])
    shapes = O.buffer_shapes(oracle_cfg(w.cfg))
    sizes = dict(zip(K.BUFFER_NAMES, K.kvq_buffer_sizes(w.cfg)))
    for n, s in sizes.items():
        if n in shapes:
            shape, dt = shapes[n]
            nbytes = int(__import__("numpy").prod(shape)) * (2 if dt.__name__ == "uint16" else 1)
            assert s == nbytes, n
        else:
            assert s == 0, n


def _bad(**kw):
    base = dict(L=1, H_kv=2, H_q=4, D=128, batch=1, max_T=64, k_fmt=K.Fmt(4, 32), v_fmt=K.Fmt(4, 32))
    base.update(kw)
    return K.Config(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(D=96), 2), (dict(H_q=3), 1), (dict(H_q=36, H_kv=2), 2), (dict(k_fmt=K.Fmt(5, 32)), 1),
    (dict(k_fmt=K.Fmt(4, 64)), 1), (dict(k_fmt=K.Fmt(4, 128, K.AXIS_CHANNEL)), 2),
    (dict(flags=K.ROTATE_K, k_fmt=K.Fmt(4, 32, K.AXIS_CHANNEL)), 2),
    (dict(flags=K.ROTATE_K | K.K_PRE_ROPE), 2), (dict(flags=128), 1), (dict(hot_window=64), 1),
    (dict(hot_window=64, k_cold=K.Fmt(2, 32), v_cold=K.Fmt(2, 32)), 2),
    (dict(page_tokens=16, n_pages=0), 1), (dict(max_T=0), 1), (dict(in_dtype=7), 1),
    (dict(k_fmt=K.Fmt(16, 32)), 1),
])
def test_validation_rejects(kw, status):
    with pytest.raises(K.KvqError) as e:
        K.kvq_validate_config(_bad(**kw))
    assert e.value.status == status
    assert K.LIB.kvq_last_error().decode() != ""


def test_workloads_validate():
    for name in W.ALL:
        K.kvq_validate_config(W.make(name).cfg)


def test_split_heuristic_fits_workspace():
    for name in W.ALL:
        cfg = W.make(name).cfg
        ws = K.kvq_workspace_bytes(cfg)
        for n in (1, cfg.L):
            s = K.kvq_decode_splits(cfg, n)
            assert 1 <= s <= 256
            units = n * cfg.batch * cfg.H_kv
            g = cfg.H_q // cfg.H_kv
            assert ws >= units * s * g * (cfg.D + 2) * 4 or s == 1


def test_split_heuristic_keeps_whole_splits():
    """Each split of the automatic policy covers at least 8 tiles of 32
    tokens of capacity, 48 for rotated layouts (or there is one split)."""
    for name in W.ALL:
        cfg = W.make(name).cfg
        tiles = (cfg.max_T + 31) // 32 + 2
        least = 48 if cfg.flags & (K.ROTATE_K | K.ROTATE_V) else 8
        for n in (1, cfg.L):
            s = K.kvq_decode_splits(cfg, n)
            assert s == 1 or tiles // s >= least, (name, n, s)
    # the headline per-layer call keeps its measured-best 19 splits
    assert K.kvq_decode_splits(W.make("llama2_7b_kivi4").cfg, 1) == 19


def test_launch_counts():
    # append: [requant to cold] + quantize (two specialized kernels or one
    # generic) + [window copy]; decode: one launch
    assert K.kvq_launch_counts(W.make("llama2_7b_kivi4").cfg) == (1 + 2, 1)
    assert K.kvq_launch_counts(W.make("mistral7b_hotcold").cfg) == (1 + 2 + 1, 1)
    assert K.kvq_launch_counts(W.make("q8_0_mha_1k").cfg) == (2, 1)
    assert K.kvq_launch_counts(W.make("ctx262k_hadamard4").cfg) == (2, 1)  # rotated kernels for K and V
    assert K.kvq_launch_counts(W.make("ctx262k_tbq4").cfg) == (2, 1)  # TBQ4 too
    # asymmetric KIVI blocks take the specialized kernels too; per-token
    # 4-bit K with 2-bit V has no specialized pair: one generic launch
    zp = _bad(flags=K.ZP_K | K.ZP_V, k_fmt=K.Fmt(4, 32, K.AXIS_CHANNEL), residual_window=128)
    assert K.kvq_launch_counts(zp) == (1 + 2, 1)
    zp8 = _bad(flags=K.ZP_V, k_fmt=K.Fmt(8, 32), v_fmt=K.Fmt(2, 32))
    assert K.kvq_launch_counts(zp8) == (2, 1)


def test_tbq4_codebook_matches_oracle():
    import numpy as np

    c, t = K.kvq_tbq4_codebook()
    oc, ot = O.tbq4_codebook()
    assert np.array_equal(np.array(c, np.float32), oc)
    assert np.array_equal(np.array(t, np.float32), ot)


@pytest.mark.parametrize("kw,ok", [
    (dict(flags=K.ROTATE_K | K.TBQ4_K, k_fmt=K.Fmt(4, 128)), True),
    (dict(flags=K.ROTATE_K | K.ROTATE_V | K.TBQ4_K | K.TBQ4_V, k_fmt=K.Fmt(4, 128), v_fmt=K.Fmt(4, 128)), True),
    (dict(flags=K.TBQ4_K, k_fmt=K.Fmt(4, 128)), False),
    (dict(flags=K.ROTATE_K | K.TBQ4_K, k_fmt=K.Fmt(4, 32)), False),
    (dict(flags=K.ROTATE_V | K.TBQ4_V, v_fmt=K.Fmt(3, 128)), False),
])
def test_tbq4_validation(kw, ok):
    if ok:
        K.kvq_validate_config(_bad(**kw))
    else:
        with pytest.raises(K.KvqError) as e:
            K.kvq_validate_config(_bad(**kw))
        assert e.value.status == 2


@pytest.mark.parametrize("kw,ok", [
    (dict(flags=K.ZP_K | K.ZP_V, k_fmt=K.Fmt(4, 32, K.AXIS_CHANNEL)), True),
    (dict(flags=K.ZP_K | K.ZP_V, k_fmt=K.Fmt(2, 32), v_fmt=K.Fmt(2, 32)), True),
    (dict(flags=K.ZP_V, k_fmt=K.Fmt(4, 32, K.AXIS_CHANNEL), hot_window=64, k_cold=K.Fmt(2, 32, K.AXIS_CHANNEL),
          v_cold=K.Fmt(2, 32)), True),
    (dict(flags=K.ZP_K, k_fmt=K.Fmt(8, 32)), False),
    (dict(flags=K.ZP_K, k_fmt=K.Fmt(3, 128)), False),
    (dict(flags=K.ZP_K, k_fmt=K.Fmt(4, 128)), False),
    (dict(flags=K.ZP_K | K.ROTATE_K, k_fmt=K.Fmt(4, 32)), False),
    (dict(flags=K.ZP_V, k_fmt=K.Fmt(4, 32, K.AXIS_CHANNEL), hot_window=64, k_cold=K.Fmt(2, 32, K.AXIS_CHANNEL),
          v_cold=K.Fmt(8, 32)), False),
])
def test_zp_validation(kw, ok):
    if ok:
        K.kvq_validate_config(_bad(**kw))
    else:
        with pytest.raises(K.KvqError) as e:
            K.kvq_validate_config(_bad(**kw))
        assert e.value.status == 2


@pytest.mark.parametrize("kw", [
    dict(flags=K.ZP_K | K.ZP_V, k_fmt=K.Fmt(4, 32, K.AXIS_CHANNEL), residual_window=128),
    dict(flags=K.ZP_K | K.ZP_V, k_fmt=K.Fmt(2, 32), v_fmt=K.Fmt(2, 32)),
    dict(flags=K.ZP_V, k_fmt=K.Fmt(4, 32, K.AXIS_CHANNEL), hot_window=64, residual_window=32,
         k_cold=K.Fmt(2, 32, K.AXIS_CHANNEL), v_cold=K.Fmt(2, 32), max_T=1000),
])
def test_zp_size_law_matches_oracle(kw):
    cfg = _bad(**kw)
    oc = oracle_cfg(cfg)
    assert K.kvq_bytes_per_token(cfg) == O.bytes_per_token(oc)
    for T in (0, 1, 31, 32, 33, 63, 64, 200, cfg.max_T):
        assert K.kvq_cache_bytes(cfg, T) == O.cache_bytes(oc, T), T
    shapes = O.buffer_shapes(oc)
    for n, sz in zip(K.BUFFER_NAMES, K.kvq_buffer_sizes(cfg)):
        if n in shapes:
            shape, dt = shapes[n]
            assert sz == int(__import__("numpy").prod(shape)) * (2 if dt.__name__ == "uint16" else 1), n


def test_step_launches():
    # one fused launch for the layouts of the tensor-core decode the step
    # files instantiate; append + decode launches for the others
    for name in ("llama2_7b_kivi4", "llama2_7b_kivi4_zp", "mistral7b_hotcold", "gqa8b_hadamard4_paged",
                 "ctx262k_hadamard4", "ctx262k_hadamard3"):
        assert K.kvq_step_launches(W.make(name).cfg) == 1, name
    for name in ("q4_0_mha_1k", "ctx262k_tbq4", "llama2_7b_kivi2_zp"):
        a, d = K.kvq_launch_counts(W.make(name).cfg)
        assert K.kvq_step_launches(W.make(name).cfg) == a + d, name


def test_stall_test_mode_bounds():
    # the failure-detection test hook takes 0 (off) .. 2^20 polls; nothing launches here
    for bad in (-1, (1 << 20) + 1):
        with pytest.raises(K.KvqError):
            K.kvq_test_force_stall(bad)
    K.kvq_test_force_stall(0)


def test_bounds_hook_needs_the_checked_build():
    # kvq_test_shrink_bounds only acts in libkvq_checked.so; the normal build refuses rows > 0
    if K.LIB_PATH.endswith("libkvq_checked.so"):
        pytest.skip("running under the checked build")
    with pytest.raises(K.KvqError):
        K.kvq_test_shrink_bounds(1)
    K.kvq_test_shrink_bounds(0)
