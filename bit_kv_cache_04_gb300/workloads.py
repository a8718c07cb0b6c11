"""Seeded synthetic workloads shaped like the pages' models.

Plain data (shapes, formats) and torch random generators only: nothing here
quantizes, attends or packs.  The same tensors feed both the CUDA path and the
CPU oracle in the tests.  Model names stand for shapes only; no weights or
datasets are involved.

Value recipes:
  * mha_1k: K, V, q ~ N(0,1) fp16; K channels 3 and 77 scaled x20.
  * llama2_7b_kivi4 / gqa8b_*: K ~ N(0,1) with round(2% * D) outlier channels
    x15 (drawn per layer and kv head), then rotary position mixing at position
    t (split-half pairs, base 1e4) so that the cache holds post-RoPE keys; V ~
    N(0,1) * sigma_t, sigma_t ~ LogNormal(0, 0.5) per token.
  * ctx262k_*: bf16 K, V ~ N(0,1), round(1% * D) outlier channels x10.
  * mistral7b_hotcold: K pre-RoPE with per-channel std ~ LogNormal(0,1),
    fixed per (layer, kv head); V ~ N(0,1).
  * ragged lengths: T_b ~ U[2048, 8192] (seeded integers).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import List, Optional

import torch

from .config import (AXIS_CHANNEL, AXIS_TOKEN, DT_BF16, DT_F16, K_PRE_ROPE, ROTATE_K, ROTATE_V, TBQ4_K, TBQ4_V,
                     ZP_K, ZP_V, Config, Fmt)

SIGN_SEED = 0x5EED5EED


@dataclass
class Workload:
    name: str
    cfg: Config
    lengths: List[int]
    values: str  # value recipe key
    extra_tokens: int = 0  # capacity headroom for decode-time appends

    def scaled(self, L=None, batch=None, T=None, lengths=None, extra=None) -> "Workload":
        """A smaller copy with the same formats and value recipe."""
        lengths = list(lengths) if lengths is not None else (
            [T] * (batch or self.cfg.batch) if T is not None else self.lengths[: (batch or self.cfg.batch)])
        b = len(lengths)
        ex = self.extra_tokens if extra is None else extra
        max_T = max(lengths) + ex
        cfg = replace(self.cfg, L=L or self.cfg.L, batch=b, max_T=max_T)
        if cfg.page_tokens:
            pages = sum(-(-(t + ex) // cfg.page_tokens) for t in lengths)
            cfg = replace(cfg, n_pages=pages + 3, max_pages_per_seq=-(-max_T // cfg.page_tokens))
        return Workload(self.name, cfg, lengths, self.values, ex)


def _ragged(batch: int, lo: int, hi: int, seed: int) -> List[int]:
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (batch,), generator=g).tolist()


def make(name: str, extra_tokens: int = 64) -> Workload:
    F16, BF16 = DT_F16, DT_BF16
    if name in ("q8_0_mha_1k", "q4_0_mha_1k"):
        b = 8 if name.startswith("q8") else 4
        cfg = Config(L=1, H_kv=4, H_q=4, D=128, batch=1, max_T=1024 + extra_tokens, in_dtype=F16,
                     k_fmt=Fmt(b, 32), v_fmt=Fmt(b, 32))
        return Workload(name, cfg, [1024], "mha_1k", extra_tokens)
    if name == "llama2_7b_kivi4":
        cfg = Config(L=32, H_kv=32, H_q=32, D=128, batch=1, max_T=32768 + extra_tokens, in_dtype=F16,
                     k_fmt=Fmt(4, 32, AXIS_CHANNEL), v_fmt=Fmt(4, 32), residual_window=128)
        return Workload(name, cfg, [32768], "llama", extra_tokens)
    if name in ("llama2_7b_kivi4_zp", "llama2_7b_kivi2_zp"):
        b = 4 if "kivi4" in name else 2
        cfg = Config(L=32, H_kv=32, H_q=32, D=128, batch=1, max_T=32768 + extra_tokens, in_dtype=F16,
                     k_fmt=Fmt(b, 32, AXIS_CHANNEL), v_fmt=Fmt(b, 32), residual_window=128, flags=ZP_K | ZP_V)
        return Workload(name, cfg, [32768], "llama", extra_tokens)
    if name == "gqa8b_hadamard4_paged":
        lengths = _ragged(16, 2048, 8192, 3)
        max_T = 8192 + extra_tokens
        pages = sum(-(-(t + extra_tokens) // 16) for t in lengths) + 3
        cfg = Config(L=32, H_kv=8, H_q=32, D=128, batch=16, max_T=max_T, in_dtype=F16,
                     k_fmt=Fmt(4, 128), v_fmt=Fmt(4, 128), flags=ROTATE_K | ROTATE_V, sign_seed=SIGN_SEED,
                     page_tokens=16, n_pages=pages, max_pages_per_seq=-(-max_T // 16))
        return Workload(name, cfg, lengths, "llama", extra_tokens)
    if name in ("ctx262k_hadamard4", "ctx262k_hadamard3", "ctx262k_tbq4"):
        b = 3 if name.endswith("3") else 4
        flags = ROTATE_K | ROTATE_V | (TBQ4_K | TBQ4_V if name.endswith("tbq4") else 0)
        cfg = Config(L=16, H_kv=4, H_q=24, D=256, batch=1, max_T=262144 + extra_tokens, in_dtype=BF16,
                     k_fmt=Fmt(b, 128), v_fmt=Fmt(b, 128), flags=flags, sign_seed=SIGN_SEED)
        return Workload(name, cfg, [262144], "ctx262k", extra_tokens)
    if name == "mistral7b_hotcold":
        cfg = Config(L=32, H_kv=8, H_q=32, D=128, batch=64, max_T=32768 + extra_tokens, in_dtype=F16,
                     k_fmt=Fmt(4, 32, AXIS_CHANNEL), v_fmt=Fmt(4, 32),
                     k_cold=Fmt(2, 32, AXIS_CHANNEL), v_cold=Fmt(2, 32),
                     hot_window=4096, residual_window=128, flags=K_PRE_ROPE, rope_theta=10000.0)
        return Workload(name, cfg, [32768] * 64, "mistral", extra_tokens)
    raise KeyError(name)


ALL = ("q8_0_mha_1k", "q4_0_mha_1k", "llama2_7b_kivi4", "gqa8b_hadamard4_paged", "ctx262k_hadamard4",
       "ctx262k_hadamard3", "mistral7b_hotcold", "ctx262k_tbq4", "llama2_7b_kivi4_zp", "llama2_7b_kivi2_zp")


def _torch_dtype(cfg: Config):
    return torch.float16 if cfg.in_dtype == DT_F16 else torch.bfloat16


def _gen(seed: int, device) -> torch.Generator:
    return torch.Generator(device=device).manual_seed(seed)


def _outlier_channels(D: int, frac: float, gen_seed: int) -> torch.Tensor:
    g = torch.Generator().manual_seed(gen_seed)
    n = max(1, round(frac * D))
    return torch.randperm(D, generator=g)[:n]


def _rotary_mix(x: torch.Tensor, pos: torch.Tensor, base: float) -> torch.Tensor:
    """Synthesis of post-RoPE keys: split-half rotary mixing at each token's
    position (the workload's keys arrive already rotated)."""
    D = x.shape[-1]
    h = D // 2
    inv = base ** (-2.0 * torch.arange(h, dtype=torch.float64, device=x.device) / D)
    ang = pos.to(torch.float64)[:, None] * inv[None, :]
    c = torch.cos(ang).to(torch.float32)[:, None, :]
    s = torch.sin(ang).to(torch.float32)[:, None, :]
    a, b = x[..., :h], x[..., h:]
    return torch.cat([a * c - b * s, a * s + b * c], dim=-1)


def kv_tokens(w: Workload, layer: int, seq: int, t0: int, t1: int, device="cpu", seed: int = 0):
    """K, V of tokens [t0, t1) of one (layer, sequence): [t1 - t0, H_kv, D] in
    the workload's input dtype.  Deterministic in (seed, layer, seq, t0, t1)."""
    cfg = w.cfg
    H, D, n = cfg.H_kv, cfg.D, t1 - t0
    key = (seed * 1_000_003 + layer * 7919 + seq * 104_729 + t0 * 31 + t1) % (2 ** 62)
    g = _gen(key, device)
    k = torch.randn((n, H, D), generator=g, device=device, dtype=torch.float32)
    v = torch.randn((n, H, D), generator=g, device=device, dtype=torch.float32)
    if w.values == "mha_1k":
        k[..., 3] *= 20.0
        k[..., 77] *= 20.0
    elif w.values == "llama":
        for h in range(H):
            ch = _outlier_channels(D, 0.02, seed * 131 + layer * 977 + h).to(device)
            k[:, h, ch] *= 15.0
        pos = torch.arange(t0, t1, device=device)
        k = _rotary_mix(k, pos, 1e4)
        sig = torch.empty((n, 1, 1), device=device).log_normal_(0.0, 0.5, generator=g)
        v = v * sig
    elif w.values == "ctx262k":
        for h in range(H):
            ch = _outlier_channels(D, 0.01, seed * 137 + layer * 983 + h).to(device)
            k[:, h, ch] *= 10.0
    elif w.values == "mistral":
        for h in range(H):
            gs = torch.Generator().manual_seed(seed * 139 + layer * 991 + h)
            std = torch.empty(D).log_normal_(0.0, 1.0, generator=gs).to(device)
            k[:, h, :] *= std
    dt = _torch_dtype(cfg)
    return k.to(dt).contiguous(), v.to(dt).contiguous()


def layer_batch(w: Workload, layer: int, starts: List[int], stops: List[int], device="cpu", seed: int = 0):
    """K, V for tokens [starts[b], stops[b]) of every sequence, concatenated in
    batch order (the layout kvq_append takes), plus cu_new."""
    ks, vs, cu = [], [], [0]
    for b, (a, e) in enumerate(zip(starts, stops)):
        k, v = kv_tokens(w, layer, b, a, e, device, seed)
        ks.append(k)
        vs.append(v)
        cu.append(cu[-1] + (e - a))
    return torch.cat(ks), torch.cat(vs), cu


def queries(w: Workload, n_layers: int, device="cpu", seed: int = 0, step: int = 0) -> torch.Tensor:
    cfg = w.cfg
    g = _gen(seed * 7 + 12345 + step * 1_000_033, device)
    q = torch.randn((n_layers, cfg.batch, cfg.H_q, cfg.D), generator=g, device=device, dtype=torch.float32)
    return q.to(_torch_dtype(cfg)).contiguous()


def page_table(w: Workload, seed: int = 0) -> Optional[torch.Tensor]:
    """A shuffled block table: every sequence gets distinct physical pages."""
    cfg = w.cfg
    if not cfg.page_tokens:
        return None
    g = torch.Generator().manual_seed(seed * 17 + 4242)
    perm = torch.randperm(cfg.n_pages, generator=g)
    table = torch.full((cfg.batch, cfg.max_pages_per_seq), -1, dtype=torch.int32)
    used = 0
    for b in range(cfg.batch):
        need = -(-min(cfg.max_T, w.lengths[b] + w.extra_tokens) // cfg.page_tokens)
        table[b, :need] = perm[used:used + need].to(torch.int32)
        used += need
    assert used <= cfg.n_pages
    return table
