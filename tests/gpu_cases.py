"""Shared driver of the GPU parity tests: the same appends on the GPU (through
the C ABI) and in the CPU oracle."""

from __future__ import annotations

import numpy as np

from oracle import kvq_oracle as O
from tests.helpers import oracle_cfg, raw16


def appended_cache(w, chunks=None, seed=0, with_oracle=True, device="cuda"):
    """Appends every layer of workload `w` in steps of `chunks` tokens per
    sequence (one multi-layer kvq_append per step).  Returns (cache,
    seq_lens (device), oracle buffers or None, block table or None)."""
    import torch

    from bit_kv_cache_04_gb300 import kvq as K
    from bit_kv_cache_04_gb300 import workloads as W

    cfg = w.cfg
    oc = oracle_cfg(cfg)
    table = W.page_table(w, seed)
    cache = K.KVCache(cfg, device, block_table=table)
    ref = O.new_buffers(oc) if with_oracle else None
    table_np = None if table is None else table.numpy()
    B, L = cfg.batch, cfg.L
    full = [[W.kv_tokens(w, l, b, 0, w.lengths[b], device, seed) for b in range(B)] for l in range(L)]
    seq_lens = torch.zeros(B, dtype=torch.int32, device=device)
    done = [0] * B
    sizes = list(chunks) if chunks else [max(w.lengths)]
    i = 0
    while any(d < t for d, t in zip(done, w.lengths)):
        step = sizes[min(i, len(sizes) - 1)] if i < len(sizes) else sizes[-1]
        i += 1
        n = [min(step, t - d) for d, t in zip(done, w.lengths)]
        cu = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
        ks = torch.stack([torch.cat([full[l][b][0][done[b]:done[b] + n[b]] for b in range(B)]) for l in range(L)])
        vs = torch.stack([torch.cat([full[l][b][1][done[b]:done[b] + n[b]] for b in range(B)]) for l in range(L)])
        cu_d = torch.as_tensor(cu, device=device)
        cache.append(0, L, ks.contiguous(), vs.contiguous(), cu_d, seq_lens, int(cu[-1]), max(n))
        cache.commit_lengths(cu_d, seq_lens)
        if with_oracle:
            for l in range(L):
                O.append(oc, ref, l, raw16(ks[l]), raw16(vs[l]), n, done, block_table=table_np)
        done = [d + x for d, x in zip(done, n)]
    torch.cuda.synchronize()
    return cache, seq_lens, ref, table_np


def gpu_buffers_as_oracle(cache, oc):
    """GPU buffers copied to the host and shaped like the oracle's."""
    shapes = O.buffer_shapes(oc)
    out = {}
    for name, arr in cache.buffer_numpy().items():
        shape, dt = shapes[name]
        out[name] = arr.view(dt).reshape(shape)
    return out


# Paged layouts of the unrotated 32-value per-token formats (their rows leave
# the per-token append kernel through the block table, one destination per
# token row): pages of 16 and of 8 tokens, a 16-bit window, asymmetric blocks.
PAGED_PER_TOKEN = {
    "q4_0_p16": ("q4_0_mha_1k", dict(page_tokens=16), [1000, 333, 129]),
    "q8_0_p8_window": ("q8_0_mha_1k", dict(page_tokens=8, residual_window=128), [700, 77, 200]),
    "q4_0_zp_p16": ("q4_0_mha_1k", dict(page_tokens=16, zp=True), [513, 31, 260]),
    "q8_0_p16_bf16": ("q8_0_mha_1k", dict(page_tokens=16, bf16=True), [640, 130, 33]),
}


def paged_workload(key):
    """The paged workload `key` of PAGED_PER_TOKEN, scaled to its lengths."""
    from dataclasses import replace

    from bit_kv_cache_04_gb300 import config as C
    from bit_kv_cache_04_gb300 import workloads as W

    name, kw, lengths = PAGED_PER_TOKEN[key]
    kw = dict(kw)
    if kw.pop("zp", False):
        kw["flags"] = C.ZP_K | C.ZP_V
    if kw.pop("bf16", False):
        kw["in_dtype"] = C.DT_BF16
    w = W.make(name)
    w = W.Workload(w.name, replace(w.cfg, **kw), w.lengths, w.values, w.extra_tokens)
    return w.scaled(lengths=lengths)
