"""Test glue: converts library configs to oracle configs, runs the same
appends on the GPU and in the oracle, and compares."""

from __future__ import annotations

import numpy as np

from oracle import kvq_oracle as O


def oracle_cfg(c) -> O.Config:
    zk, zv = bool(c.flags & 32), bool(c.flags & 64)  # the library's asymmetric-block flags

    def f(x, zp):
        return None if x is None else O.Fmt(x.bits, x.group, x.axis, zp)

    return O.Config(L=c.L, H_kv=c.H_kv, H_q=c.H_q, D=c.D, batch=c.batch, max_T=c.max_T, in_dtype=c.in_dtype,
                    k_fmt=f(c.k_fmt, zk), v_fmt=f(c.v_fmt, zv), k_cold=f(c.k_cold, zk), v_cold=f(c.v_cold, zv),
                    hot_window=c.hot_window, residual_window=c.residual_window, flags=c.flags,
                    rope_theta=c.rope_theta, sign_seed=c.sign_seed, page_tokens=c.page_tokens,
                    n_pages=c.n_pages, max_pages_per_seq=c.max_pages_per_seq)


def raw16(t) -> np.ndarray:
    """A torch fp16/bf16 tensor as raw uint16 bits on the host."""
    import torch

    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def rel_err(out, ref) -> float:
    """max over heads of ||out - ref||_inf / ||ref||_inf (heads with a zero
    reference compare absolutely)."""
    out = np.asarray(out, np.float64)
    ref = np.asarray(ref, np.float64)
    num = np.max(np.abs(out - ref), axis=-1)
    den = np.max(np.abs(ref), axis=-1)
    r = np.where(den > 0, num / np.where(den > 0, den, 1), num)
    return float(np.max(r)) if r.size else 0.0


def codes_differ(cfg: O.Config, gpu: dict, ref: dict):
    """(elements compared, elements whose code differs, max |code diff|,
    blocks whose scale differs) over every quantized buffer."""
    total = diff = maxd = sdiff = 0
    for name in gpu:
        if name.endswith("resid"):
            continue
        which = name[0]
        tier_cold = name.endswith("cold")
        fmt = (cfg.k_cold if which == "k" else cfg.v_cold) if tier_cold else (cfg.k_fmt if which == "k" else cfg.v_fmt)
        bb = O.block_bytes(fmt.bits, fmt.group, fmt.zp)
        a = gpu[name].reshape(-1, bb)
        b = ref[name].reshape(-1, bb)
        if fmt.zp:
            sa, _, ca = O.decode_blocks_zp(a, fmt.bits, fmt.group)
            sb, _, cb = O.decode_blocks_zp(b, fmt.bits, fmt.group)
        else:
            sa, ca = O.decode_blocks(a, fmt.bits, fmt.group)
            sb, cb = O.decode_blocks(b, fmt.bits, fmt.group)
        d = np.abs(ca.astype(np.int32) - cb.astype(np.int32))
        total += d.size
        diff += int(np.count_nonzero(d))
        maxd = max(maxd, int(d.max()) if d.size else 0)
        sdiff += int(np.count_nonzero(sa.view(np.uint16) != sb.view(np.uint16)))
    return total, diff, maxd, sdiff
