"""GPU parity against the CPU oracle on seeded inputs, at sizes the oracle
finishes in seconds (several tiles and a ragged tail per sequence).

* Packed codes and scales: byte-identical buffers (the GPU follows the
  format's fp32 op order, rotated formats included).
* Decode attention: max over heads of ||o - o_ref||_inf / ||o_ref||_inf
  <= 2e-3 against fp64 attention over the same dequantized cache (the oracle
  decodes the GPU's own bytes).
* kvq_dequantize: equal to the oracle's dequantization of the GPU bytes
  (exact for unrotated formats; rotated ones within fp32 transform rounding).
"""

import numpy as np
import pytest

from oracle import kvq_oracle as O
from tests.gpu_cases import PAGED_PER_TOKEN, appended_cache, gpu_buffers_as_oracle, paged_workload
from tests.helpers import codes_differ, oracle_cfg, raw16, rel_err

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from bit_kv_cache_04_gb300 import kvq as K  # noqa: E402
from bit_kv_cache_04_gb300 import workloads as W  # noqa: E402

TOL = 2e-3

CASES = {
    "q8_0_mha_1k": dict(),
    "q4_0_mha_1k": dict(),
    "llama2_7b_kivi4": dict(L=2, lengths=[700, 333, 129]),
    "gqa8b_hadamard4_paged": dict(L=2, lengths=[300, 77, 129, 16]),
    "ctx262k_hadamard4": dict(L=2, lengths=[1000]),
    "ctx262k_hadamard3": dict(L=2, lengths=[777]),
    "mistral7b_hotcold": dict(L=1, lengths=[4500, 4390, 200]),
}


def _workload(name):
    w = W.make(name)
    kw = CASES[name]
    return w.scaled(**kw) if kw else w


def _decode(cache, w, seq_lens, n_layers=None, layer0=0, splits=0, seed=0):
    cfg = w.cfg
    n = n_layers or cfg.L
    q = W.queries(w, n, "cuda", seed)
    out = torch.full((n, cfg.batch, cfg.H_q, cfg.D), float("nan"), dtype=torch.float32, device="cuda")
    cache.decode(layer0, n, q, seq_lens, out, num_splits=splits)
    torch.cuda.synchronize()
    return q, out


@pytest.mark.parametrize("name", sorted(CASES))
def test_append_bytes_identical(name):
    w = _workload(name)
    cache, seq_lens, ref, _ = appended_cache(w)
    got = gpu_buffers_as_oracle(cache, oracle_cfg(w.cfg))
    assert cache.device_status() == 0
    for n in ref:
        if not np.array_equal(got[n], ref[n]):
            total, diff, maxd, sdiff = codes_differ(oracle_cfg(w.cfg), {n: got[n]}, {n: ref[n]}) \
                if not n.endswith("resid") else (0, -1, -1, -1)
            pytest.fail(f"{n}: bytes differ (codes {diff}/{total}, max |dc| {maxd}, scales {sdiff})")


@pytest.mark.parametrize("name", sorted(CASES))
def test_decode_matches_fp64_oracle(name):
    w = _workload(name)
    cache, seq_lens, _, table = appended_cache(w, with_oracle=False)
    oc = oracle_cfg(w.cfg)
    q, out = _decode(cache, w, seq_lens)
    assert torch.isfinite(out).all()
    bufs = gpu_buffers_as_oracle(cache, oc)
    ref = O.decode_attention(oc, bufs, 0, w.cfg.L, raw16(q), w.lengths, block_table=table)
    err = rel_err(out.cpu().numpy(), ref)
    assert err <= TOL, err


@pytest.mark.parametrize("name", ["llama2_7b_kivi4", "mistral7b_hotcold", "gqa8b_hadamard4_paged", "q4_0_mha_1k"])
def test_bulk_and_incremental_append_agree(name):
    w = _workload(name)
    bulk, sl_b, _, table = appended_cache(w, with_oracle=False)
    inc, sl_i, ref, _ = appended_cache(w, chunks=[257, 1, 1, 33, 31, 1, 64, 500, 3])
    oc = oracle_cfg(w.cfg)
    gb, gi = gpu_buffers_as_oracle(bulk, oc), gpu_buffers_as_oracle(inc, oc)
    for n in ref:
        assert np.array_equal(gi[n], ref[n]), n
    # live state (what decode reads) is the same after bulk or incremental append
    for l in range(w.cfg.L):
        for b in range(w.cfg.batch):
            x = O.dequantize(oc, gb, l, b, w.lengths[b], block_table=table)
            y = O.dequantize(oc, gi, l, b, w.lengths[b], block_table=table)
            assert np.array_equal(x[0], y[0]) and np.array_equal(x[1], y[1])
    _, o1 = _decode(bulk, w, sl_b)
    _, o2 = _decode(inc, w, sl_i)
    assert torch.equal(o1, o2)


@pytest.mark.parametrize("key", sorted(PAGED_PER_TOKEN))
def test_paged_per_token_formats(key):
    w = paged_workload(key)
    oc = oracle_cfg(w.cfg)
    for chunks in (None, [257, 1, 1, 33, 31, 1, 64, 500, 3]):
        cache, seq_lens, ref, table = appended_cache(w, chunks=chunks)
        assert cache.device_status() == 0
        got = gpu_buffers_as_oracle(cache, oc)
        for n in ref:
            assert np.array_equal(got[n], ref[n]), (n, chunks)
    q, out = _decode(cache, w, seq_lens)
    ref_o = O.decode_attention(oc, got, 0, w.cfg.L, raw16(q), w.lengths, block_table=table)
    assert rel_err(out.cpu().numpy(), ref_o) <= TOL


@pytest.mark.parametrize("name", ["llama2_7b_kivi4", "ctx262k_hadamard4", "mistral7b_hotcold"])
def test_split_count_does_not_matter(name):
    w = _workload(name)
    cache, seq_lens, _, _ = appended_cache(w, with_oracle=False)
    _, base = _decode(cache, w, seq_lens, splits=1)
    for s in (2, 5, 16):
        _, o = _decode(cache, w, seq_lens, splits=s)
        assert rel_err(o.cpu().numpy(), base.cpu().numpy()) < 1e-5, s
    # one layer in 48 chunks per unit (the workspace holds up to 64 for one
    # layer): units of 32 chunks or more merge in two levels
    _, o = _decode(cache, w, seq_lens, n_layers=1, splits=48)
    assert rel_err(o.cpu().numpy(), base[:1].cpu().numpy()) < 1e-5


# Per-layer calls whose chunk plan takes one whole wave of resident blocks,
# more than batch x splits (the grid is widened): equal lengths split evenly
# over the budget's share of the grid, ragged lengths planned by tile count.
# Both agree with the fp64 oracle, and with one split per unit up to the
# order of the fp32 sums: each split rounds its probabilities' fp16 hi / lo
# parts against its own running maximum, and over the 256 groups of an
# 8192-token unit the two orders differ by ~3e-5 (the full-size test allows
# 1e-4 for up to 1024 groups on the same grounds).
WAVE_CASES = [("gqa8b_hadamard4_paged", [8192] * 3), ("gqa8b_hadamard4_paged", [8192, 3000, 500]),
              ("mistral7b_hotcold", [8192] * 3), ("mistral7b_hotcold", [5000, 2500, 700, 64, 3000]),
              ("ctx262k_hadamard4", [8192] * 3)]


@pytest.mark.parametrize("name,lengths", WAVE_CASES)
def test_one_wave_budget_matches_one_split_and_oracle(name, lengths):
    w = W.make(name).scaled(L=1, lengths=lengths)
    cache, seq_lens, _, table = appended_cache(w, with_oracle=False)
    q, base = _decode(cache, w, seq_lens, splits=1)
    _, out = _decode(cache, w, seq_lens)
    assert cache.device_status() == 0
    assert rel_err(out.cpu().numpy(), base.cpu().numpy()) < 1e-4
    oc = oracle_cfg(w.cfg)
    ref = O.decode_attention(oc, gpu_buffers_as_oracle(cache, oc), 0, 1, raw16(q), w.lengths, block_table=table)
    assert rel_err(out.cpu().numpy(), ref) <= TOL


def test_per_layer_calls_equal_multi_layer_call():
    w = _workload("llama2_7b_kivi4")
    cache, seq_lens, _, _ = appended_cache(w, with_oracle=False)
    q, out = _decode(cache, w, seq_lens)
    for l in range(w.cfg.L):
        o = torch.empty_like(out[l:l + 1])
        cache.decode(l, 1, q[l:l + 1].contiguous(), seq_lens, o)
        torch.cuda.synchronize()
        assert rel_err(o.cpu().numpy(), out[l:l + 1].cpu().numpy()) < 1e-5


@pytest.mark.parametrize("name", sorted(CASES))
def test_dequantize_matches_oracle(name):
    w = _workload(name)
    cache, seq_lens, _, table = appended_cache(w, with_oracle=False)
    oc = oracle_cfg(w.cfg)
    bufs = gpu_buffers_as_oracle(cache, oc)
    rotated = bool(w.cfg.flags & (K.ROTATE_K | K.ROTATE_V))
    for b in range(w.cfg.batch):
        T = w.lengths[b]
        for t0, t1 in ((0, T), (T // 3, T // 3 + 45)):
            t1 = min(t1, T)
            if t1 <= t0:
                continue
            k = torch.empty((t1 - t0, w.cfg.H_kv, w.cfg.D), dtype=torch.float32, device="cuda")
            v = torch.empty_like(k)
            cache.dequantize(w.cfg.L - 1, b, t0, t1, seq_lens, k, v)
            rk, rv = O.dequantize(oc, bufs, w.cfg.L - 1, b, T, t0, t1, block_table=table)
            for g_, r_ in ((k, rk), (v, rv)):
                g_ = g_.cpu().numpy().astype(np.float64)
                if rotated:
                    assert np.max(np.abs(g_ - r_)) <= 1e-5 * max(1.0, np.max(np.abs(r_)))
                else:
                    assert np.array_equal(g_, r_)
    assert cache.device_status() == 0


def test_empty_and_single_token_sequences():
    w = W.make("q4_0_mha_1k").scaled(lengths=[1, 0, 5])
    cache, seq_lens, _, _ = appended_cache(w, with_oracle=False)
    q, out = _decode(cache, w, seq_lens)
    out = out.cpu().numpy()
    assert np.all(out[0, 1] == 0)
    oc = oracle_cfg(w.cfg)
    bufs = gpu_buffers_as_oracle(cache, oc)
    K1, V1 = O.dequantize(oc, bufs, 0, 0, 1)
    for h in range(w.cfg.H_q):
        assert np.allclose(out[0, 0, h], V1[0, h], rtol=1e-6, atol=1e-6)


def test_device_status_bits():
    w = W.make("q4_0_mha_1k").scaled(lengths=[40, 10], extra=0)
    cache, seq_lens, _, _ = appended_cache(w, with_oracle=False)
    cfg = w.cfg
    # an append past capacity is skipped and flagged
    k = torch.zeros((1, 2, cfg.H_kv, cfg.D), dtype=torch.float16, device="cuda")
    cu = torch.tensor([0, 2, 2], dtype=torch.int32, device="cuda")
    before = cache.buffer_numpy()
    cache.append(0, 1, k, k, cu, seq_lens, 2, 2)
    assert cache.device_status() & K.DEV_CAPACITY
    after = cache.buffer_numpy()
    assert all(np.array_equal(before[n], after[n]) for n in before)
    cache.clear_status()
    assert cache.device_status() == 0
    # a dequantize range beyond the current length is flagged, nothing written
    kk = torch.full((5, cfg.H_kv, cfg.D), 7.0, device="cuda")
    cache.dequantize(0, 1, 8, 13, seq_lens, kk, kk.clone())
    assert cache.device_status() & K.DEV_RANGE
    assert torch.all(kk == 7.0)


def test_bad_page_id_is_flagged_not_faulted():
    w = _workload("gqa8b_hadamard4_paged")
    cache, seq_lens, _, _ = appended_cache(w, with_oracle=False)
    cache.block_table[1, 0] = w.cfg.n_pages + 5
    cache.block_table[2, 1] = -1
    _decode(cache, w, seq_lens)
    assert cache.device_status() & K.DEV_PAGE


def test_host_validation_launches_nothing():
    w = W.make("q4_0_mha_1k")
    cache = K.KVCache(w.cfg, "cuda")
    q = torch.zeros((1, 1, 4, 128), dtype=torch.float16, device="cuda")
    out = torch.zeros((1, 1, 4, 128), dtype=torch.float32, device="cuda")
    sl = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(K.KvqError):
        cache.decode(0, 2, q, sl, out)  # layers beyond L
    with pytest.raises(K.KvqError):
        cache.decode(0, 1, q, sl, out, num_splits=1000)
    # misaligned input rows are refused before any launch
    kv = torch.zeros((1, 2 * 4 * 128 + 8), dtype=torch.float16, device="cuda")
    k_bad = kv[:, 1:1 + 4 * 128].view(1, 1, 4, 128)
    cu = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    with pytest.raises(K.KvqError):
        cache.append(0, 1, k_bad, k_bad, cu, sl, 1, 1)
    torch.cuda.synchronize()
    assert cache.device_status() == 0
