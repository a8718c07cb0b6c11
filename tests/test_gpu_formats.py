"""Byte parity of quantize-on-append for every bit width, block axis, input
dtype and head dim of the 32-value block formats (and of TBQ4 blocks: norm +
Lloyd-Max indices, where decode and dequantize are checked too), on two kinds
of input:

* exact ties: every block's absolute maximum is qmax * s with s a power of two
  (so s16 = s exactly) and every other value is (k + 1/2) s, so every code is
  decided by round-half-to-even.  The maxima sit where token index and
  channel index agree mod 32, so per-token blocks (32 channels of a token) and
  per-channel blocks (one channel over 32 tokens) both hold one.  One kv head
  uses s = 2^-20, a subnormal fp16 scale;
* seeded N(0, 1) values with a few large channels.

* for the asymmetric (scale + zero point) blocks, exact half steps between
  each block's minimum and maximum with a power-of-two range / (2^b - 1);
* for the asymmetric blocks also blocks whose unclamped codes leave
  [0, 2^b - 1] (the kernels quantize those with the clamp): ranges of a few
  steps of 2^-24 (fp16 scales that round down), bf16 values beyond the fp16
  zero point's range, and single infinities.  The test checks on the CPU that
  such blocks occur.

Each case appends in two calls (a bulk prefix, then a ragged remainder) and
compares every packed byte with the oracle.
"""

import zlib

import numpy as np
import pytest

from oracle import kvq_oracle as O
from tests.helpers import codes_differ, oracle_cfg, raw16, rel_err

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from bit_kv_cache_04_gb300 import kvq as K  # noqa: E402

CH, TOK = K.AXIS_CHANNEL, K.AXIS_TOKEN

# (name, D, dtype, k_fmt, v_fmt, k_cold, v_cold, hot_window, residual_window[, flags])
CASES = [
    ("t8_f16", 128, K.DT_F16, K.Fmt(8, 32), K.Fmt(8, 32), None, None, 0, 0),
    ("t8_bf16_d256", 256, K.DT_BF16, K.Fmt(8, 32), K.Fmt(8, 32), None, None, 0, 16),
    ("t4_bf16", 128, K.DT_BF16, K.Fmt(4, 32), K.Fmt(4, 32), None, None, 0, 0),
    ("t3_f16", 128, K.DT_F16, K.Fmt(3, 32), K.Fmt(3, 32), None, None, 0, 0),
    ("t2_bf16", 128, K.DT_BF16, K.Fmt(2, 32), K.Fmt(2, 32), None, None, 0, 0),
    ("kivi4_bf16", 128, K.DT_BF16, K.Fmt(4, 32, CH), K.Fmt(4, 32), None, None, 0, 128),
    ("kivi2_f16_d256", 256, K.DT_F16, K.Fmt(2, 32, CH), K.Fmt(2, 32), None, None, 0, 64),
    ("tiers_bf16", 128, K.DT_BF16, K.Fmt(4, 32, CH), K.Fmt(4, 32), K.Fmt(2, 32, CH), K.Fmt(2, 32), 64, 32),
    ("tiers_f16_d256", 256, K.DT_F16, K.Fmt(4, 32, CH), K.Fmt(4, 32), K.Fmt(2, 32, CH), K.Fmt(2, 32), 96, 0),
    # asymmetric blocks (scale + zero point)
    ("zp_kivi4_f16", 128, K.DT_F16, K.Fmt(4, 32, CH), K.Fmt(4, 32), None, None, 0, 128, K.ZP_K | K.ZP_V),
    ("zp_t2_bf16", 128, K.DT_BF16, K.Fmt(2, 32), K.Fmt(2, 32), None, None, 0, 0, K.ZP_K | K.ZP_V),
    ("zp_tiers_f16", 128, K.DT_F16, K.Fmt(4, 32, CH), K.Fmt(4, 32), K.Fmt(2, 32, CH), K.Fmt(2, 32), 64, 32,
     K.ZP_K | K.ZP_V),
    ("zp_v_only_d256", 256, K.DT_F16, K.Fmt(4, 32, CH), K.Fmt(2, 32), None, None, 0, 32, K.ZP_V),
    ("zp_kivi2_f16", 128, K.DT_F16, K.Fmt(2, 32, CH), K.Fmt(2, 32), None, None, 0, 64, K.ZP_K | K.ZP_V),
    ("zp_tiers_rope_f16", 128, K.DT_F16, K.Fmt(4, 32, CH), K.Fmt(4, 32), K.Fmt(2, 32, CH), K.Fmt(2, 32), 64, 32,
     K.ZP_K | K.ZP_V | K.K_PRE_ROPE),
    ("zp_kivi4_rope_f16", 128, K.DT_F16, K.Fmt(4, 32, CH), K.Fmt(4, 32), None, None, 0, 0,
     K.ZP_K | K.ZP_V | K.K_PRE_ROPE),
]

LENGTHS = [301, 160, 33]
PREFIX = [200, 64, 0]


def _inputs(kind, n_tok, H, D, bits, gen, zp=False, bf16=False):
    """[n_tok, H, D] input values (float64) for one tensor; token index is the
    position within the sequence."""
    if kind == "clamp" and zp:
        # heads in turn: tiny integer steps, large magnitudes (with a few
        # infinities), N(0, 1); W is constant over every block of either axis
        t = torch.arange(n_tok).view(-1, 1, 1)
        c = torch.arange(D).view(1, 1, -1)
        hh = torch.arange(H).view(1, -1, 1)
        W = (16 + ((t // 32) * 5 + (c // 32) * 11 + hh * 3) % 40).double()
        k = torch.floor(torch.rand((n_tok, H, D), generator=gen, dtype=torch.float64) * (W + 1))
        sign = torch.where(((t // 32) + (c // 32) + hh) % 2 == 0, 1.0, -1.0).double()
        tiny = (k - 7) * 2.0 ** -24
        big = sign * ((2.0 ** 16 + k * 512) if bf16 else (61440 + k * 32))
        inf = torch.zeros((n_tok, H, D), dtype=torch.float64)
        inf = torch.where(((t % 97) == 5) & ((c % 53) == 1), float("inf"), inf)
        inf = torch.where(((t % 89) == 7) & ((c % 59) == 2), float("-inf"), inf)
        big = torch.where(inf != 0, inf, big)
        mode = (hh % 3).expand(n_tok, H, D)
        rnd = torch.randn((n_tok, H, D), generator=gen, dtype=torch.float64)
        return torch.where(mode == 0, tiny, torch.where(mode == 1, big, rnd))
    if kind == "ties" and zp:
        # asymmetric ties: every block holds its minimum -off*s (where token
        # and channel agree mod 32, shifted by one) and its maximum
        # (qlev - off)*s, so the scale is s and the zero -off*s exactly; every
        # other value is (k + 1/2 - off)*s, an exact half step
        qlev = (1 << bits) - 1
        off = qlev // 2
        k = torch.randint(0, qlev, (n_tok, H, D), generator=gen, dtype=torch.int64).double() + 0.5
        t = torch.arange(n_tok).view(-1, 1, 1)
        c = torch.arange(D).view(1, 1, -1)
        hi = ((t % 32) == (c % 32)).expand(n_tok, H, D)
        lo = ((t % 32) == ((c + 1) % 32)).expand(n_tok, H, D)
        x = torch.where(hi, float(qlev), torch.where(lo, 0.0, k)) - off
        s = torch.tensor([2.0 ** (-3 * (h % 3)) for h in range(H)], dtype=torch.float64).view(1, H, 1)
        s[0, -1, 0] = 2.0 ** -20
        return x * s
    if kind == "ties":
        qmax = (1 << (bits - 1)) - 1
        k = torch.randint(-qmax, qmax, (n_tok, H, D), generator=gen, dtype=torch.int64).double() + 0.5
        t = torch.arange(n_tok).view(-1, 1, 1)
        c = torch.arange(D).view(1, 1, -1)
        diag = (t % 32) == (c % 32)
        sign = torch.where(torch.rand((n_tok, H, D), generator=gen) < 0.5, -1.0, 1.0).double()
        x = torch.where(diag.expand(n_tok, H, D), sign * qmax, k)
        s = torch.tensor([2.0 ** (-3 * (h % 3)) for h in range(H)], dtype=torch.float64).view(1, H, 1)
        s[0, -1, 0] = 2.0 ** -20
        return x * s
    x = torch.randn((n_tok, H, D), generator=gen, dtype=torch.float64)
    x[..., 5] *= 12
    x[..., D - 9] *= 30
    return x


def _case_tensors(kind, cfg, lengths, which, gen):
    bits = (cfg.k_fmt if which == 0 else cfg.v_fmt).bits
    zp = bool(cfg.flags & (K.ZP_K if which == 0 else K.ZP_V))
    dt = torch.float16 if cfg.in_dtype == K.DT_F16 else torch.bfloat16
    return [_inputs(kind, T, cfg.H_kv, cfg.D, bits, gen, zp, dt == torch.bfloat16).to(dt) for T in lengths]


def _blocks_needing_clamp(x, fmt):
    """How many full 32-value blocks of x ([T, H, D] 16-bit) along the
    format's axis have an unclamped code outside [0, 2^b - 1] (numpy fp32, the
    quantizer's op order; a coverage count, not a parity check)."""
    a = x.float().numpy()
    if fmt.axis == CH:
        n = a.shape[0] // 32 * 32
        a = a[:n].reshape(n // 32, 32, *a.shape[1:]).transpose(0, 2, 3, 1)
    else:
        a = a.reshape(*a.shape[:-1], a.shape[-1] // 32, 32)
    qlev = np.float32((1 << fmt.bits) - 1)
    with np.errstate(all="ignore"):
        mn = a.min(-1) + np.float32(0.0)
        s = np.minimum((a.max(-1) - mn) / qlev, np.float32(65504)).astype(np.float16).astype(np.float32)
        z = np.clip(mn, -65504, 65504).astype(np.float16).astype(np.float32)
        r = np.rint((a - z[..., None]) / s[..., None])
    out = ((r < 0) | (r > qlev)) & (s[..., None] != 0)
    return int(out.any(-1).sum())


KIND_CASES = [(c, k) for c in CASES for k in ("ties", "random")] + [(c, "clamp") for c in CASES if len(c) > 9]


@pytest.mark.parametrize("case,kind", KIND_CASES, ids=[f"{c[0]}-{k}" for c, k in KIND_CASES])
def test_append_bytes_match_oracle(case, kind):
    name, D, dtype, kf, vf, kc, vc, hot, R = case[:9]
    flags = case[9] if len(case) > 9 else 0
    # asymmetric cases also decode, with three query heads per kv head
    cfg = K.Config(L=1, H_kv=3, H_q=9 if flags else 3, D=D, batch=len(LENGTHS), max_T=max(LENGTHS) + 32,
                   in_dtype=dtype, k_fmt=kf, v_fmt=vf, k_cold=kc, v_cold=vc, hot_window=hot, residual_window=R,
                   flags=flags)
    oc = oracle_cfg(cfg)
    gen = torch.Generator().manual_seed(zlib.crc32(f"{name}/{kind}".encode()))
    ks = _case_tensors(kind, cfg, LENGTHS, 0, gen)
    vs = _case_tensors(kind, cfg, LENGTHS, 1, gen)
    if kind == "clamp":
        for which, xs, f in ((0, ks, kf), (1, vs, vf)):
            if flags & (K.ZP_K if which == 0 else K.ZP_V):
                assert sum(_blocks_needing_clamp(x, f) for x in xs) > 0, (name, which)
    cache = K.KVCache(cfg, "cuda")
    ref = O.new_buffers(oc)
    seq_lens = torch.zeros(cfg.batch, dtype=torch.int32, device="cuda")
    done = [0] * cfg.batch
    for step in (PREFIX, [T - p for T, p in zip(LENGTHS, PREFIX)]):
        kk = torch.cat([ks[b][done[b]:done[b] + step[b]] for b in range(cfg.batch)])
        vv = torch.cat([vs[b][done[b]:done[b] + step[b]] for b in range(cfg.batch)])
        cu = np.concatenate([[0], np.cumsum(step)]).astype(np.int32)
        cu_d = torch.as_tensor(cu, device="cuda")
        cache.append(0, 1, kk[None].cuda().contiguous(), vv[None].cuda().contiguous(), cu_d, seq_lens,
                     int(cu[-1]), max(step))
        cache.commit_lengths(cu_d, seq_lens)
        O.append(oc, ref, 0, raw16(kk), raw16(vv), step, done)
        done = [d + x for d, x in zip(done, step)]
    torch.cuda.synchronize()
    assert cache.device_status() == 0
    shapes = O.buffer_shapes(oc)
    bufs = {}
    for n, arr in cache.buffer_numpy().items():
        shape, dt = shapes[n]
        got = arr.view(dt).reshape(shape)
        bufs[n] = got
        if not np.array_equal(got, ref[n]):
            total, diff, maxd, sdiff = codes_differ(oc, {n: got}, {n: ref[n]}) \
                if not n.endswith("resid") else (0, -1, -1, -1)
            pytest.fail(f"{name}/{kind} {n}: bytes differ (codes {diff}/{total}, max |dc| {maxd}, scales {sdiff})")
    if flags and kind != "clamp":  # asymmetric blocks: decode over the GPU's bytes against fp64 attention
        dtq = torch.float16 if dtype == K.DT_F16 else torch.bfloat16
        q = torch.randn((1, cfg.batch, cfg.H_q, D), generator=gen).to(dtq).cuda()
        out = torch.full((1, cfg.batch, cfg.H_q, D), float("nan"), dtype=torch.float32, device="cuda")
        cache.decode(0, 1, q, seq_lens, out)
        torch.cuda.synchronize()
        o_ref = O.decode_attention(oc, bufs, 0, 1, raw16(q), LENGTHS)
        assert rel_err(out.cpu().numpy(), o_ref) <= 2e-3


# ---- TBQ4 (norm + Lloyd-Max codebook) -------------------------------------------

TBQ4_CASES = [
    ("tbq4_f16_d128", 128, K.DT_F16, 0, 32),          # window: the generic decode kernel
    ("tbq4_f16_d128_mma", 128, K.DT_F16, 7, 0),        # the tensor-core decode, D = 128
    ("tbq4_bf16_d256_seed", 256, K.DT_BF16, 0x5EED, 0),  # the tensor-core decode, D = 256
    # blocks outside the fast quotient's bounds (bytes only)
    ("tbq4_bf16_d256_edge", 256, K.DT_BF16, 3, 0, "edge"),
    ("tbq4_f16_d128_edge", 128, K.DT_F16, 5, 0, "edge"),
]


def _tbq4_edge(n_tok, H, D, gen, bf16):
    """[n_tok, H, D] values whose 128-value blocks take every branch of the
    TBQ4 quantizer, by token index mod 6: N(0, 1); all zeros (zero norm);
    a few units of 2^-24 (tiny norms, some rotated values exactly 0); huge
    values (the norm saturates at 65504); N(0, 1) with one infinity; 1 and +-1
    in channels 10, 11 and beta in channel 70, zeros elsewhere: where the
    sign flips make the first butterfly cancel, half the rotated values are
    +-beta c (beta = 2^-110 for bf16: far below 2^-100 next to values near 1)."""
    x = torch.randn((n_tok, H, D), generator=gen, dtype=torch.float64)
    kind = (torch.arange(n_tok) % 6).view(-1, 1, 1).expand(n_tok, H, D)
    tiny = torch.randint(-3, 4, (n_tok, H, D), generator=gen).double() * 2.0 ** -24
    huge = x * 1e30 if bf16 else (x * 30000.0).clamp(-65504.0, 65504.0)
    one_inf = torch.where((torch.arange(D) == 17).view(1, 1, -1), float("inf"), x)
    c = torch.arange(D).view(1, 1, -1)
    sgn = torch.where(torch.rand((n_tok, H, 1), generator=gen) < 0.5, -1.0, 1.0).double()
    beta = 2.0 ** (-110 if bf16 else -24)
    cancel = torch.where(c == 10, 1.0, torch.where(c == 11, sgn, torch.where(c == 70, beta, 0.0)))
    out = torch.where(kind == 1, 0.0, x)
    out = torch.where(kind == 2, tiny, out)
    out = torch.where(kind == 3, huge, out)
    out = torch.where(kind == 4, one_inf, out)
    return torch.where(kind == 5, cancel.expand(n_tok, H, D), out)


@pytest.mark.parametrize("case", TBQ4_CASES, ids=[c[0] for c in TBQ4_CASES])
def test_tbq4_bytes_decode_and_dequantize(case):
    name, D, dtype, seed, R = case[:5]
    edge = len(case) > 5
    flags = K.ROTATE_K | K.ROTATE_V | K.TBQ4_K | K.TBQ4_V
    cfg = K.Config(L=1, H_kv=3, H_q=6, D=D, batch=len(LENGTHS), max_T=max(LENGTHS) + 32, in_dtype=dtype,
                   k_fmt=K.Fmt(4, 128), v_fmt=K.Fmt(4, 128), residual_window=R, flags=flags, sign_seed=seed)
    oc = oracle_cfg(cfg)
    gen = torch.Generator().manual_seed(zlib.crc32(name.encode()))
    dt = torch.float16 if dtype == K.DT_F16 else torch.bfloat16
    if edge:
        ks = [_tbq4_edge(T, cfg.H_kv, D, gen, dt == torch.bfloat16).to(dt) for T in LENGTHS]
        vs = [_tbq4_edge(T, cfg.H_kv, D, gen, dt == torch.bfloat16).to(dt) for T in LENGTHS]
    else:
        ks = [_inputs("random", T, cfg.H_kv, D, 4, gen).to(dt) for T in LENGTHS]
        vs = [_inputs("random", T, cfg.H_kv, D, 4, gen).to(dt) for T in LENGTHS]
    cache = K.KVCache(cfg, "cuda")
    ref = O.new_buffers(oc)
    seq_lens = torch.zeros(cfg.batch, dtype=torch.int32, device="cuda")
    done = [0] * cfg.batch
    for step in (PREFIX, [T - p for T, p in zip(LENGTHS, PREFIX)]):
        kk = torch.cat([ks[b][done[b]:done[b] + step[b]] for b in range(cfg.batch)])
        vv = torch.cat([vs[b][done[b]:done[b] + step[b]] for b in range(cfg.batch)])
        cu = np.concatenate([[0], np.cumsum(step)]).astype(np.int32)
        cu_d = torch.as_tensor(cu, device="cuda")
        cache.append(0, 1, kk[None].cuda().contiguous(), vv[None].cuda().contiguous(), cu_d, seq_lens,
                     int(cu[-1]), max(step))
        cache.commit_lengths(cu_d, seq_lens)
        O.append(oc, ref, 0, raw16(kk), raw16(vv), step, done)
        done = [d + x for d, x in zip(done, step)]
    torch.cuda.synchronize()
    assert cache.device_status() == 0
    shapes = O.buffer_shapes(oc)
    got = {}
    for n, arr in cache.buffer_numpy().items():
        shape, dtn = shapes[n]
        got[n] = arr.view(dtn).reshape(shape)
        if not np.array_equal(got[n], ref[n]):
            total, diff, maxd, sdiff = codes_differ(oc, {n: got[n]}, {n: ref[n]}) \
                if not n.endswith("resid") else (0, -1, -1, -1)
            pytest.fail(f"{name} {n}: bytes differ (codes {diff}/{total}, max |dc| {maxd}, scales {sdiff})")
    if edge:
        return
    if R == 0:
        # the GPU's indices against the plain reading of the norm (fp64 sum,
        # no summation order): within 1 on at most 1e-4 of the elements
        signs = O.hadamard_signs(seed)
        total = differ = 0
        for name_, xs in (("k_main", ks), ("v_main", vs)):
            for b, T in enumerate(LENGTHS):
                rows = np.moveaxis(got[name_][0, b, :, :T], 0, 1).reshape(T, cfg.H_kv, D // 128, 66)
                gi = O.decode_blocks(rows, 4, 128)[1].astype(np.int64) + 8
                y = O.rotate_f32(O.input_to_f32(raw16(xs[b]), dtype), *signs).reshape(T, cfg.H_kv, D // 128, 128)
                d = np.abs(gi - O.tbq4_quantize_f64norm(y)[1].astype(np.int64))
                assert d.max() <= 1, (name, name_, b)
                total += d.size
                differ += int(np.count_nonzero(d))
        assert differ <= 1e-4 * total, (name, differ, total)
    # decode over the GPU's own bytes, against fp64 attention
    q = torch.randn((1, cfg.batch, cfg.H_q, D), generator=gen).to(dt).cuda()
    out = torch.full((1, cfg.batch, cfg.H_q, D), float("nan"), dtype=torch.float32, device="cuda")
    cache.decode(0, 1, q, seq_lens, out)
    torch.cuda.synchronize()
    o_ref = O.decode_attention(oc, got, 0, 1, raw16(q), LENGTHS)
    assert rel_err(out.cpu().numpy(), o_ref) <= 2e-3
    # dequantize (original domain; the GPU undoes the rotation in fp32)
    for b, T in enumerate(LENGTHS):
        kd = torch.empty((T, cfg.H_kv, D), dtype=torch.float32, device="cuda")
        vd = torch.empty_like(kd)
        cache.dequantize(0, b, 0, T, seq_lens, kd, vd)
        torch.cuda.synchronize()
        rk, rv = O.dequantize(oc, got, 0, b, T)
        for g_, r_ in ((kd, rk), (vd, rv)):
            diff = np.abs(g_.cpu().numpy().astype(np.float64) - r_)
            assert diff.max() <= 1e-5 * max(1.0, np.abs(r_).max()), (name, b, diff.max())
