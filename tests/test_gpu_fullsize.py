"""Parity at the workloads' full sizes, in the launch configuration bench.py
times (one bulk kvq_append per layer, one multi-layer kvq_decode_attention
with the default split count), checked on sampled outputs the oracle computes
one by one:

* packed bytes of sampled rows (the oracle re-quantizes the same source
  tokens, regenerated from the seeded generator);
* decode outputs of sampled (layer, sequence, query head) triples against
  fp64 attention over the GPU's own dequantized cache, max relative error
  <= 2e-3.
"""

import numpy as np
import pytest

from oracle import kvq_oracle as O
from tests.helpers import oracle_cfg, raw16, rel_err

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from bit_kv_cache_04_gb300 import kvq as K  # noqa: E402
from bit_kv_cache_04_gb300 import workloads as W  # noqa: E402

TOL = 2e-3


def _full_cache(name):
    w = W.make(name, extra_tokens=16)
    cfg = w.cfg
    table = W.page_table(w)
    cache = K.KVCache(cfg, "cuda", block_table=table)
    seq_lens = torch.zeros(cfg.batch, dtype=torch.int32, device="cuda")
    for layer in range(cfg.L):
        ks, vs, cu = W.layer_batch(w, layer, [0] * cfg.batch, w.lengths, "cuda")
        cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
        cache.append(layer, 1, ks[None], vs[None], cu_d, seq_lens, cu[-1], max(w.lengths))
        del ks, vs
    cu_all = torch.tensor([0] + list(np.cumsum(w.lengths)), dtype=torch.int32, device="cuda")
    cache.commit_lengths(cu_all, seq_lens)
    torch.cuda.synchronize()
    assert cache.device_status() == 0
    return w, cache, seq_lens, (None if table is None else table.numpy())


def _layer_view(cache, oc, layer):
    """Host copies of one layer of every buffer, shaped like the oracle's
    buffers but with a layer dimension of 1 (index it with layer 0)."""
    shapes = O.buffer_shapes(oc)
    out = {}
    for name, t in cache.buffers.items():
        if t is None:
            continue
        shape, dt = shapes[name]
        per_layer = t.numel() // shape[0]
        chunk = t[layer * per_layer:(layer + 1) * per_layer].cpu().numpy().view(dt)
        out[name] = chunk.reshape((1,) + tuple(shape[1:]))
    return out


SAMPLES = {
    "q8_0_mha_1k": [(0, 0, 0), (0, 0, 3)],
    "q4_0_mha_1k": [(0, 0, 1), (0, 0, 2)],
    "llama2_7b_kivi4": [(0, 0, 0), (17, 0, 9), (31, 0, 31)],
    "gqa8b_hadamard4_paged": [(0, 0, 0), (13, 7, 21), (31, 15, 31)],
    "ctx262k_hadamard4": [(0, 0, 0), (15, 0, 23)],
    "ctx262k_hadamard3": [(0, 0, 5), (15, 0, 18)],
    "mistral7b_hotcold": [(0, 0, 0), (20, 33, 14), (31, 63, 31)],
    "ctx262k_tbq4": [(0, 0, 2), (15, 0, 20)],
    "llama2_7b_kivi4_zp": [(0, 0, 0), (31, 0, 17)],
    "llama2_7b_kivi2_zp": [(0, 0, 3), (31, 0, 30)],
}


@pytest.mark.parametrize("name", W.ALL)
def test_full_size_decode_and_codes(name):
    w, cache, seq_lens, table = _full_cache(name)
    cfg = w.cfg
    oc = oracle_cfg(cfg)
    q = W.queries(w, cfg.L, "cuda", seed=5)
    out = torch.full((cfg.L, cfg.batch, cfg.H_q, cfg.D), float("nan"), dtype=torch.float32, device="cuda")
    cache.decode(0, cfg.L, q, seq_lens, out)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    assert cache.device_status() == 0
    # the sampled layers again as single-layer calls (the split planner's
    # chunks, and the two-level merge where a unit has 32 or more): the same
    # outputs up to the order of the fp32 sums, which over up to 1024 groups
    # of a sequence stays within 1024 * 2^-24 ~ 6e-5
    for layer in sorted({x[0] for x in SAMPLES[name]}):
        o1 = torch.full_like(out[layer:layer + 1], float("nan"))
        cache.decode(layer, 1, q[layer:layer + 1].contiguous(), seq_lens, o1)
        torch.cuda.synchronize()
        assert cache.device_status() == 0
        assert rel_err(o1.cpu().numpy(), out[layer:layer + 1].cpu().numpy()) < 1e-4, (layer, K.kvq_decode_splits(cfg, 1))
    qh = raw16(q)
    g = cfg.H_q // cfg.H_kv
    lengths = [w.lengths[b] for b in range(cfg.batch)]
    for layer, seq, hq in SAMPLES[name]:
        bufs = _layer_view(cache, oc, layer)
        ref = O.decode_attention(oc, bufs, 0, 1, qh[layer:layer + 1], lengths, block_table=table,
                                 which=[(0, seq, hq)])
        err = rel_err(out[layer, seq, hq].cpu().numpy()[None], ref[0, seq, hq][None])
        assert err <= TOL, (layer, seq, hq, err)
        # codes: the oracle appends this kv head's whole sequence on its own
        # and must hold the same values for the first and last 64 tokens
        kvh = hq // g
        T = w.lengths[seq]
        one = O.Config(**{**oc.__dict__, "L": 1, "batch": 1, "H_kv": 1, "H_q": g, "page_tokens": 0, "n_pages": 0,
                          "max_pages_per_seq": 0})
        ks, vs = W.kv_tokens(w, layer, seq, 0, T, "cuda")
        ob = O.new_buffers(one)
        O.append(one, ob, 0, raw16(ks[:, kvh:kvh + 1]), raw16(vs[:, kvh:kvh + 1]), [T], [0])
        del ks, vs
        for t0, t1 in ((0, min(64, T)), (max(0, T - 64), T)):
            gk, gv = O.dequantize(oc, bufs, 0, seq, T, t0, t1, block_table=table, heads=[kvh])
            rk, rv = O.dequantize(one, ob, 0, 0, T, t0, t1)
            assert np.array_equal(gk, rk) and np.array_equal(gv, rv), (layer, seq, t0)
