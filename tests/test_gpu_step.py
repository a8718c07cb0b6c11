"""The decode step (kvq_decode_step): one new token appended to every sequence
and decode attention over the grown cache, in one launch for the layouts of
the tensor-core decode (the blocks that own the tiles the token changes write
them first).  Each case runs many consecutive steps from a bulk-appended
prefix, so the window hands groups to the packed tier and, with tiers, groups
move from hot to cold, at every split count tried.  Checked:

* after every step the outputs equal those of the unfused path (kvq_append,
  length commit, kvq_decode_attention) bit for bit, and no status bit is set;
* at the end both caches hold the same bytes, equal to the oracle's cache of
  the same tokens appended one at a time;
* the last step's attention matches fp64 attention over that cache
  (<= 2e-3, as the decode tests).
"""

import numpy as np
import pytest

from oracle import kvq_oracle as O
from tests.gpu_cases import appended_cache, gpu_buffers_as_oracle
from tests.helpers import oracle_cfg, raw16, rel_err

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from bit_kv_cache_04_gb300 import kvq as K  # noqa: E402
from bit_kv_cache_04_gb300 import workloads as W  # noqa: E402

STEPS = 40

# (workload, scaled shape, split counts); the lengths put group flushes and
# (hot/cold) demotions inside the 40 steps
CASES = [
    ("llama2_7b_kivi4", dict(L=2, lengths=[290, 161, 130], extra=48), (0, 5)),
    ("llama2_7b_kivi4_zp", dict(L=1, lengths=[300, 133], extra=48), (0, 3)),
    ("mistral7b_hotcold", dict(L=1, lengths=[4330, 4301, 150], extra=48), (0, 7)),
    ("gqa8b_hadamard4_paged", dict(L=2, lengths=[300, 77, 129, 16], extra=48), (0, 4)),
    ("ctx262k_hadamard4", dict(L=1, lengths=[500], extra=48), (0, 6)),
    ("ctx262k_hadamard3", dict(L=1, lengths=[333], extra=48), (0,)),
    # layouts the step runs as append + decode launches
    ("q4_0_mha_1k", dict(L=1, lengths=[200], extra=48), (0,)),
    ("ctx262k_tbq4", dict(L=1, lengths=[300], extra=48), (0,)),
    ("llama2_7b_kivi2_zp", dict(L=1, lengths=[250, 40], extra=48), (0,)),
]


@pytest.mark.parametrize("name,shape,splits", CASES, ids=[c[0] for c in CASES])
def test_decode_step_matches_unfused_and_oracle(name, shape, splits):
    w = W.make(name).scaled(**shape)
    cfg = w.cfg
    oc = oracle_cfg(cfg)
    B, L = cfg.batch, cfg.L
    fused = K.kvq_step_launches(cfg) == 1
    assert fused == (name not in ("q4_0_mha_1k", "ctx262k_tbq4", "llama2_7b_kivi2_zp"))
    for ns in splits:
        cache_f, seq_f, ref, table = appended_cache(w)
        cache_u, seq_u, _, _ = appended_cache(w, with_oracle=False)
        cu_one = torch.arange(B + 1, dtype=torch.int32, device="cuda")
        done = list(w.lengths)
        out_f = torch.empty((L, B, cfg.H_q, cfg.D), dtype=torch.float32, device="cuda")
        out_u = torch.empty_like(out_f)
        for s in range(STEPS):
            kv = [[W.kv_tokens(w, l, b, done[b], done[b] + 1, "cuda", seed=0) for b in range(B)] for l in range(L)]
            k_new = torch.stack([torch.cat([kv[l][b][0] for b in range(B)]) for l in range(L)]).contiguous()
            v_new = torch.stack([torch.cat([kv[l][b][1] for b in range(B)]) for l in range(L)]).contiguous()
            q = W.queries(w, L, "cuda", seed=1, step=s)
            out_f.fill_(float("nan"))
            out_u.fill_(float("nan"))
            cache_f.decode_step(0, L, k_new, v_new, q, seq_f, out_f, num_splits=ns)
            cache_f.commit_lengths(cu_one, seq_f)
            cache_u.append(0, L, k_new, v_new, cu_one, seq_u, B, 1)
            cache_u.commit_lengths(cu_one, seq_u)
            cache_u.decode(0, L, q, seq_u, out_u, num_splits=ns)
            torch.cuda.synchronize()
            assert torch.equal(out_f, out_u), (name, ns, s, (out_f - out_u).abs().max().item())
            for l in range(L):
                O.append(oc, ref, l, raw16(k_new[l]), raw16(v_new[l]), [1] * B, done, block_table=table)
            done = [d + 1 for d in done]
        assert cache_f.device_status() == 0 and cache_u.device_status() == 0
        assert torch.equal(seq_f, seq_u) and seq_f.cpu().tolist() == done
        got_f = gpu_buffers_as_oracle(cache_f, oc)
        got_u = gpu_buffers_as_oracle(cache_u, oc)
        for n in got_f:
            assert np.array_equal(got_f[n], got_u[n]), (name, ns, n)
            assert np.array_equal(got_f[n], ref[n]), (name, ns, n)
        o_ref = O.decode_attention(oc, got_f, 0, L, raw16(q), done, block_table=table)
        assert rel_err(out_f.cpu().numpy(), o_ref) <= 2e-3


def test_step_on_an_empty_sequence():
    """A step on a sequence of length 0 attends to its one new token: the
    output is that token's value."""
    w = W.make("llama2_7b_kivi4").scaled(L=1, lengths=[0, 0], extra=40)
    cfg = w.cfg
    cache = K.KVCache(cfg, "cuda")
    seq = torch.zeros(2, dtype=torch.int32, device="cuda")
    k_new = torch.randn((1, 2, cfg.H_kv, cfg.D), device="cuda").half()
    v_new = torch.randn((1, 2, cfg.H_kv, cfg.D), device="cuda").half()
    q = W.queries(w, 1, "cuda")
    out = torch.empty((1, 2, cfg.H_q, cfg.D), dtype=torch.float32, device="cuda")
    cache.decode_step(0, 1, k_new, v_new, q, seq, out)
    torch.cuda.synchronize()
    g = cfg.H_q // cfg.H_kv
    want = v_new.float().repeat_interleave(g, dim=2)
    assert torch.equal(out, want)
    assert cache.device_status() == 0


def test_step_errors_are_refused_or_flagged():
    """Bad arguments are refused on the host; a step past capacity and a new
    token on a bad page set status bits and write nothing out of range."""
    w = W.make("llama2_7b_kivi4").scaled(L=1, lengths=[40], extra=8)
    cfg = w.cfg
    cache, seq, _, _ = appended_cache(w, with_oracle=False)
    q = W.queries(w, 1, "cuda")
    out = torch.empty((1, 1, cfg.H_q, cfg.D), dtype=torch.float32, device="cuda")
    kn = torch.zeros((1, 1, cfg.H_kv, cfg.D), dtype=torch.float16, device="cuda")
    with pytest.raises(K.KvqError):
        cache.decode_step(0, 1, None, kn, q, seq, out)
    flat = torch.zeros(1 + cfg.H_kv * cfg.D, dtype=torch.float16, device="cuda")
    with pytest.raises(K.KvqError):  # 2-byte aligned rows
        cache.decode_step(0, 1, flat[1:].view(1, 1, cfg.H_kv, cfg.D), kn, q, seq, out)
    with pytest.raises(K.KvqError):
        cache.decode_step(0, 2, kn, kn, q, seq, out)  # layers beyond L
    # past capacity: flagged, the cache unchanged
    full = torch.full((1,), cfg.max_T, dtype=torch.int32, device="cuda")
    before = cache.buffer_numpy()
    cache.decode_step(0, 1, kn, kn, q, full, out)
    torch.cuda.synchronize()
    assert cache.device_status() != 0
    after = cache.buffer_numpy()
    assert all(np.array_equal(before[n], after[n]) for n in before)
    # paged layout: the page of sequence 0's new token (position 32, page 2) is out of range
    w2 = W.make("gqa8b_hadamard4_paged").scaled(L=1, lengths=[32, 16], extra=32)
    c2 = w2.cfg
    cache2, seq2, _, _ = appended_cache(w2, with_oracle=False)
    cache2.block_table[0, 2] = c2.n_pages + 3
    kn2 = torch.zeros((1, 2, c2.H_kv, c2.D), dtype=torch.float16, device="cuda")
    q2 = W.queries(w2, 1, "cuda")
    out2 = torch.empty((1, 2, c2.H_q, c2.D), dtype=torch.float32, device="cuda")
    cache2.decode_step(0, 1, kn2, kn2, q2, seq2, out2)
    torch.cuda.synchronize()
    assert cache2.device_status() & K.DEV_PAGE
