"""Plain CPU oracle for the quantized KV cache.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` import this module.
The product path (the CUDA library and its Python binding) never calls it, and
this module imports nothing from the product.

What it computes, step by step, with the page each step follows:

* Size law (nalar.dev "Kuantisasi KV Cache dengan Error Budget yang Eksplisit",
  section "Ukuran cache mengikuti jumlah elemen tersimpan dan bit width": the
  cache holds 2*L*T*H_kv*D scalars; trefon.com "Matematyka cache KV", section
  "Bajty na token" and the format table of "Przyklad: model 27B przy 262K").
* Block formats: an fp16 scale followed by G*b/8 bytes of packed codes
  (trefon.com, format table: Q8_0 34 B/32, Q4_0 18 B/32, 66 B/128, 50 B/128).
* Absmax quantization in fp32 with the op order: fp32 amax, scale = amax/qmax
  rounded to fp16, code = rint(x / float(scale)), clamp.  Keys are grouped per
  channel over token groups and values per token (troisinh.com "KV Cache
  Quantization", section "Tai sao Key va Value lai khac nhau?"; trefon.com,
  section "Dlaczego cache trudniej skwantyzowac niz wagi").
* Optional randomized Walsh-Hadamard rotation of each 128-element block:
  sign flip, transform, sign flip, orthonormal (trefon.com, section "Jak
  4-bitowemu cache to uchodzi: najpierw obrot").
* A recent window kept at 16 bits and a hot/cold 4-bit/2-bit split
  (nalar.dev, section "Evaluasi harus memisahkan..."; troisinh.com, section
  "Mixed Precision").
* Keys stored before RoPE and rotated on the fly with split-half RoPE
  (troisinh.com, "RoPE - Cai bay tinh vi"; lehuy.net "NexusQuant", section
  "Cac mo hinh duoc ho tro": split-half pairs).
* TBQ4 (trefon.com, section "Jak 4-bitowemu cache to uchodzi: najpierw
  obrot"): after the rotation, a 128-value block is stored as its L2 norm
  (fp16) and, per value, the 4-bit index of the nearest of the 16 Lloyd-Max
  centroids for N(0, sigma^2), sigma = 1/sqrt(128); the centroids come from
  Lloyd's algorithm run here in fp64 (S. P. Lloyd, "Least squares
  quantization in PCM", 1982; J. Max, 1960) and the lookup table holds them
  rounded to fp16.
* Asymmetric ("scale and zero point") blocks, the next step the pages name
  for KIVI's 2/4-bit cache (nalar.dev, section "Granularitas kuantisasi...":
  low-bit codes need a scale and sometimes a zero point; troisinh.com
  "Asymmetric Quantization"): the block stores its fp16 scale and its fp16
  minimum, codes c in [0, 2^b - 1] and x = c * scale + zero.
* Decode attention, the plain definition in fp64: s_i = q.k_i / sqrt(D),
  p = softmax(s), output = sum_i p_i v_i (nalar.dev, sections "Error pada key
  mengubah input softmax" and "Error pada value masuk setelah attention
  probability").

Readings where the pages are silent (the plainest reading in each case):
symmetric codes in [-qmax, qmax] with qmax = 2^(b-1)-1; half-to-even rounding;
fp16 scale saturating at 65504; a zero scale gives all-zero codes; nibble and
bit order little-endian and element-ascending; 3-bit values packed eight to a
24-bit little-endian word; the 2-bit block is 10 B/32; GQA maps query head h
to kv head h // (H_q/H_kv); an empty sequence attends to nothing and yields 0.

Byte layouts of the cache buffers (the same contract the CUDA library keeps;
written here independently from its description):

* per-token block row: D/G blocks of one token and kv head, back to back;
* per-channel group row: D blocks (one per channel, channel-ascending) that
  each cover the G tokens of one token group;
* main tier, contiguous: [L][batch][H_kv][capacity][row], capacity = max_T
  rounded up to a multiple of 32 tokens (per-token) or ceil(max_T/G) groups;
* main tier, paged (per-token formats only): [L][pages][H_kv][page_tokens][row],
  page = block_table[seq][t // page_tokens];
* two tiers: the hot tier is a ring (per-channel: W/G + 1 group slots; per-token:
  W + G token slots) and the cold tier an absolute array;
* 16-bit window: ring [L][batch][H_kv][R + Gamma][D] of raw input-dtype bits,
  slot = t mod (R + Gamma), Gamma = the per-channel group (1 without one).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, Optional, Tuple

import numpy as np

AXIS_TOKEN = 0
AXIS_CHANNEL = 1

ROTATE_K = 1
ROTATE_V = 2
K_PRE_ROPE = 4
TBQ4_K = 8
TBQ4_V = 16

DT_F16 = 0
DT_BF16 = 1

QMAX = {8: 127, 4: 7, 3: 3, 2: 1}

# 1/sqrt(128) rounded to fp32 (bits 0x3DB504F3): the scale of the orthonormal
# 128-point transform, applied once after the butterflies.
HADAMARD_SCALE_F32 = np.float32(2.0 ** -3.5)

M64 = (1 << 64) - 1


# ----------------------------------------------------------------------------
# Formats and configuration
# ----------------------------------------------------------------------------


@dataclass(frozen=True)
class Fmt:
    """A block format: `bits` per code and `group` values per fp16 scale.

    axis = AXIS_TOKEN: a block spans `group` consecutive channels of one token.
    axis = AXIS_CHANNEL: a block spans one channel over `group` consecutive tokens.
    bits = 16 is accepted by the size law only (plain 16-bit storage).
    """

    bits: int
    group: int
    axis: int = AXIS_TOKEN
    zp: bool = False  # asymmetric blocks: fp16 scale + fp16 zero (the block minimum), codes 0..2^b-1


@dataclass
class Config:
    L: int
    H_kv: int
    H_q: int
    D: int
    batch: int
    max_T: int
    in_dtype: int = DT_F16
    k_fmt: Fmt = Fmt(4, 32)
    v_fmt: Fmt = Fmt(4, 32)
    k_cold: Optional[Fmt] = None
    v_cold: Optional[Fmt] = None
    hot_window: int = 0
    residual_window: int = 0
    flags: int = 0
    rope_theta: float = 10000.0
    sign_seed: int = 0
    page_tokens: int = 0
    n_pages: int = 0
    max_pages_per_seq: int = 0


def block_bytes(bits: int, group: int, zp: bool = False) -> int:
    """One block: fp16 scale (2 B) + group*bits/8 bytes of codes (trefon.com
    format table); asymmetric blocks add an fp16 zero point (2 B).  bits == 16
    means plain 16-bit values with no scale."""
    if bits == 16:
        return 2 * group
    return 2 + (2 if zp else 0) + group * bits // 8


def unit_tokens(cfg: Config) -> int:
    """Gamma: the token granularity of quantization (the per-channel group,
    or 1 when every format is per-token)."""
    g = 1
    for f in (cfg.k_fmt, cfg.v_fmt):
        if f.axis == AXIS_CHANNEL:
            g = max(g, f.group)
    return g


def q_end(cfg: Config, T: int) -> int:
    """End of the quantized prefix: tokens [q_end, T) stay in the 16-bit
    window (nalar.dev: a recent window at higher precision is part of the
    representation)."""
    gam = unit_tokens(cfg)
    R = cfg.residual_window
    if T <= R:
        return 0
    return ((T - R) // gam) * gam


def c_end(cfg: Config, T: int) -> int:
    """End of the cold (low-bit) tier: the hot tier keeps the W most recent
    quantized tokens, rounded to whole groups (troisinh.com, MixKVQ)."""
    W = cfg.hot_window
    if W <= 0:
        return 0
    gam = unit_tokens(cfg)
    qe = q_end(cfg, T)
    if qe <= W:
        return 0
    return ((qe - W) // gam) * gam


def ring_slots(cfg: Config) -> int:
    gam = unit_tokens(cfg)
    if cfg.residual_window == 0 and gam == 1:
        return 0
    return cfg.residual_window + gam


# ----------------------------------------------------------------------------
# Size law
# ----------------------------------------------------------------------------


def fmt_bytes(fmt: Fmt, n_tokens: int, D: int) -> int:
    """Bytes that hold n_tokens of one kv head in `fmt`."""
    bb = block_bytes(fmt.bits, fmt.group, fmt.zp)
    if fmt.axis == AXIS_TOKEN:
        return n_tokens * (D // fmt.group) * bb
    assert n_tokens % fmt.group == 0
    return (n_tokens // fmt.group) * D * bb


def scalars(L: int, T: int, H_kv: int, D: int) -> int:
    """2 * L * T * H_kv * D: stored scalars of one sequence (nalar.dev)."""
    return 2 * L * T * H_kv * D


def bytes_per_token(cfg: Config) -> int:
    """Steady-state bytes per token over all layers, K and V, in the format
    that holds most tokens of a long sequence (the cold tier when there is
    one).  Scales and packing count (nalar.dev: compare actual bytes per
    token, not nominal bits)."""
    kf = cfg.k_cold if cfg.hot_window > 0 else cfg.k_fmt
    vf = cfg.v_cold if cfg.hot_window > 0 else cfg.v_fmt
    total = 0
    for f in (kf, vf):
        bb = block_bytes(f.bits, f.group, f.zp)
        if f.axis == AXIS_TOKEN:
            total += (cfg.D // f.group) * bb
        else:
            assert (cfg.D * bb) % f.group == 0
            total += cfg.D * bb // f.group
    return cfg.L * cfg.H_kv * total


def cache_bytes(cfg: Config, T: int) -> int:
    """Exact bytes the representation keeps for one sequence of T tokens:
    cold tier + hot (or only) tier + 16-bit window, all layers, K and V."""
    c, q = c_end(cfg, T), q_end(cfg, T)
    per_head = 0
    if cfg.hot_window > 0:
        per_head += fmt_bytes(cfg.k_cold, c, cfg.D) + fmt_bytes(cfg.v_cold, c, cfg.D)
    per_head += fmt_bytes(cfg.k_fmt, q - c, cfg.D) + fmt_bytes(cfg.v_fmt, q - c, cfg.D)
    per_head += 2 * (T - q) * cfg.D * 2
    return cfg.L * cfg.H_kv * per_head


# ----------------------------------------------------------------------------
# Number formats
# ----------------------------------------------------------------------------


def f16_bits_to_f32(u16: np.ndarray) -> np.ndarray:
    return np.asarray(u16, np.uint16).view(np.float16).astype(np.float32)


def bf16_bits_to_f32(u16: np.ndarray) -> np.ndarray:
    """bf16 is the top half of an fp32: widening is exact."""
    return (np.asarray(u16, np.uint16).astype(np.uint32) << 16).view(np.float32)


def input_to_f32(u16: np.ndarray, in_dtype: int) -> np.ndarray:
    if in_dtype == DT_F16:
        return f16_bits_to_f32(u16)
    return bf16_bits_to_f32(u16)


# ----------------------------------------------------------------------------
# Randomized Walsh-Hadamard rotation (trefon.com, "najpierw obrot")
# ----------------------------------------------------------------------------


def splitmix64_stream(seed: int, n: int) -> list:
    """n outputs of SplitMix64 (Steele, Lea and Flood, 2014) from `seed`."""
    out = []
    state = seed & M64
    for _ in range(n):
        state = (state + 0x9E3779B97F4A7C15) & M64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
        out.append(z ^ (z >> 31))
    return out


def hadamard_signs(seed: int) -> Tuple[np.ndarray, np.ndarray]:
    """The two +-1 vectors of the randomized transform.  Seed 0 gives all +1
    (the plain Sylvester transform); otherwise bit i of the 128-bit string made
    of SplitMix64 outputs 0,1 (resp. 2,3), least significant bit first, set
    means -1."""
    if seed == 0:
        one = np.ones(128, np.float32)
        return one, one.copy()
    w = splitmix64_stream(seed, 4)
    d = []
    for pair in ((w[0], w[1]), (w[2], w[3])):
        bits = [(pair[i // 64] >> (i % 64)) & 1 for i in range(128)]
        d.append(np.where(np.array(bits) == 1, -1.0, 1.0).astype(np.float32))
    return d[0], d[1]


def sylvester(n: int = 128) -> np.ndarray:
    """Sylvester Hadamard matrix in natural order: H[i, j] = (-1)^popcount(i & j)."""
    i = np.arange(n)
    pc = np.vectorize(lambda v: bin(v).count("1"))(i[:, None] & i[None, :])
    return np.where(pc % 2 == 0, 1, -1).astype(np.int64)


def fwht_f32(x: np.ndarray) -> np.ndarray:
    """Unnormalized fast Walsh-Hadamard transform of the last axis (length 128)
    in fp32, radix-2 stages with strides 1, 2, 4, ..., 64 in that order; each
    stage maps (a, b) = (x[i], x[i+h]) to (a + b, a - b)."""
    y = np.asarray(x, np.float32)
    lead = y.shape[:-1]
    h = 1
    while h < 128:
        y = y.reshape(*lead, 128 // (2 * h), 2, h)
        a = y[..., 0, :]
        b = y[..., 1, :]
        y = np.stack([a + b, a - b], axis=-2).reshape(*lead, 128)
        h *= 2
    return y


def rotate_f32(x: np.ndarray, d1: np.ndarray, d2: np.ndarray) -> np.ndarray:
    """Forward rotation of every 128-chunk of the last axis, fp32:
    y = d2 * (FWHT(d1 * x) * (1/sqrt(128)))."""
    x = np.asarray(x, np.float32)
    D = x.shape[-1]
    xs = x.reshape(*x.shape[:-1], D // 128, 128)
    y = fwht_f32(xs * d1) * HADAMARD_SCALE_F32
    y = y * d2
    return y.reshape(x.shape).astype(np.float32)


def rotation_matrix_f64(d1: np.ndarray, d2: np.ndarray) -> np.ndarray:
    """R = diag(d2) H diag(d1) / sqrt(128) in fp64 (orthonormal)."""
    H = sylvester(128).astype(np.float64)
    return (d2.astype(np.float64)[:, None] * H * d1.astype(np.float64)[None, :]) / math.sqrt(128.0)


def unrotate_f64(y: np.ndarray, d1: np.ndarray, d2: np.ndarray) -> np.ndarray:
    """Inverse rotation (R^T) of every 128-chunk of the last axis, fp64."""
    R = rotation_matrix_f64(d1, d2)
    y = np.asarray(y, np.float64)
    D = y.shape[-1]
    ys = y.reshape(*y.shape[:-1], D // 128, 128)
    x = ys @ R  # row vector times R == (R^T y^T)^T
    return x.reshape(y.shape)


def rotate_f64(x: np.ndarray, d1: np.ndarray, d2: np.ndarray) -> np.ndarray:
    R = rotation_matrix_f64(d1, d2)
    x = np.asarray(x, np.float64)
    D = x.shape[-1]
    xs = x.reshape(*x.shape[:-1], D // 128, 128)
    return (xs @ R.T).reshape(x.shape)


# ----------------------------------------------------------------------------
# Absmax block quantization (fp32, stated op order)
# ----------------------------------------------------------------------------


def quantize(x: np.ndarray, bits: int) -> Tuple[np.ndarray, np.ndarray]:
    """Quantize blocks along the last axis.

    amax = max|x| (fp32); s32 = amax / qmax (IEEE fp32 division);
    s16 = fp16 round-to-nearest-even of min(s32, 65504);
    code = clamp(rint(x / float(s16)), -qmax, qmax), all codes 0 when s16 == 0.
    Returns (s16 as float16 [...], codes as int8 [..., G]).
    """
    x = np.asarray(x, np.float32)
    qmax = np.float32(QMAX[bits])
    amax = np.max(np.abs(x), axis=-1)
    s32 = (amax / qmax).astype(np.float32)
    s16 = np.minimum(s32, np.float32(65504.0)).astype(np.float16)
    sf = s16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        r = np.rint(np.divide(x, sf, dtype=np.float32))
    r = np.where(sf == 0, np.float32(0), r)
    codes = np.clip(r, -qmax, qmax).astype(np.int8)
    return s16, codes


def quantize_zp(x: np.ndarray, bits: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Asymmetric blocks along the last axis, fp32 op order:

    mn, mx = min x, max x; qlev = 2^b - 1; s32 = (mx - mn) / qlev;
    s16 = fp16(min(s32, 65504)); z16 = fp16(mn clipped to +-65504), a zero
    minimum stored as +0 (the minimum is a value; -0 and +0 are the same one);
    code = clamp(rint((x - float(z16)) / float(s16)), 0, qlev), all codes 0
    when s16 == 0.  Returns (s16, z16 as float16 [...], codes uint8 [..., G]).
    """
    x = np.asarray(x, np.float32)
    qlev = np.float32((1 << bits) - 1)
    mn = (np.min(x, axis=-1) + np.float32(0.0)).astype(np.float32)  # -0 + +0 = +0
    mx = np.max(x, axis=-1)
    s32 = ((mx - mn).astype(np.float32) / qlev).astype(np.float32)
    s16 = np.minimum(s32, np.float32(65504.0)).astype(np.float16)
    z16 = np.clip(mn, np.float32(-65504.0), np.float32(65504.0)).astype(np.float16)
    sf = s16.astype(np.float32)[..., None]
    zf = z16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        r = np.rint(np.divide((x - zf).astype(np.float32), sf, dtype=np.float32))
    r = np.where(sf == 0, np.float32(0), r)
    codes = np.clip(r, 0, qlev).astype(np.uint8)
    return s16, z16, codes


def dequantize_zp_f32(s16: np.ndarray, z16: np.ndarray, codes: np.ndarray) -> np.ndarray:
    """code * scale + zero in fp32: the product is exact, the sum rounds once."""
    sf = np.asarray(s16, np.float16).astype(np.float32)[..., None]
    zf = np.asarray(z16, np.float16).astype(np.float32)[..., None]
    return (codes.astype(np.float32) * sf + zf).astype(np.float32)


def dequantize_zp_f64(s16: np.ndarray, z16: np.ndarray, codes: np.ndarray) -> np.ndarray:
    """code * scale + zero, exact in fp64."""
    return (codes.astype(np.float64) * np.asarray(s16, np.float16).astype(np.float64)[..., None]
            + np.asarray(z16, np.float16).astype(np.float64)[..., None])


_PACK_BIAS = {8: 0, 4: 8, 3: 4, 2: 2}


def dequantize_f32(s16: np.ndarray, codes: np.ndarray) -> np.ndarray:
    """code * scale in fp32; exact, as |code| < 2^8 and the scale has 11 bits."""
    return codes.astype(np.float32) * np.asarray(s16, np.float16).astype(np.float32)[..., None]


def dequantize_f64(s16: np.ndarray, codes: np.ndarray) -> np.ndarray:
    return codes.astype(np.float64) * np.asarray(s16, np.float16).astype(np.float64)[..., None]


# ----------------------------------------------------------------------------
# TBQ4: L2 norm + Lloyd-Max codebook of the rotated block
# ----------------------------------------------------------------------------


def _normal_pdf(z: float) -> float:
    return math.exp(-0.5 * z * z) / math.sqrt(2.0 * math.pi)


def _normal_upper(z: float) -> float:
    """P(Z > z) for a standard normal Z."""
    return 0.5 * math.erfc(z / math.sqrt(2.0))


def lloyd_max_normal(levels: int = 16, sigma: float = 1.0 / math.sqrt(128.0), tol: float = 1e-15,
                     max_iter: int = 100000):
    """Lloyd's algorithm for the minimum mean-square-error quantizer with
    `levels` (even) points for N(0, sigma^2), in fp64.

    Alternates the two optimality conditions until the centroids stop moving
    (max change <= tol, in units of sigma): each threshold is the midpoint of
    its two neighbouring centroids; each centroid is the conditional mean of
    the distribution between its thresholds, E[Z | a < Z < b] =
    (pdf(a) - pdf(b)) / (P(Z > a) - P(Z > b)).  The density is symmetric, so
    the positive half is iterated (middle threshold 0) and mirrored.
    Returns (centroids [levels], thresholds [levels - 1], iterations), fp64,
    ascending.
    """
    half = levels // 2
    c = [(j + 0.5) * 0.5 for j in range(half)]
    it = 0
    for it in range(1, max_iter + 1):
        t = [0.0] + [(c[j] + c[j + 1]) / 2.0 for j in range(half - 1)]
        new = []
        for j in range(half):
            a = t[j]
            upper_b = _normal_upper(t[j + 1]) if j + 1 < half else 0.0
            pdf_b = _normal_pdf(t[j + 1]) if j + 1 < half else 0.0
            new.append((_normal_pdf(a) - pdf_b) / (_normal_upper(a) - upper_b))
        moved = max(abs(x - y) for x, y in zip(new, c))
        c = new
        if moved <= tol:
            break
    pos = np.array(c, np.float64) * sigma
    cent = np.concatenate([-pos[::-1], pos])
    thr = (cent[:-1] + cent[1:]) / 2.0
    return cent, thr, it


_CODEBOOK = None


def tbq4_codebook() -> Tuple[np.ndarray, np.ndarray]:
    """The format's tables, as fp32 arrays: the 16-entry centroid table holds
    the fp64 Lloyd-Max centroids rounded once to fp16 (the decoder's lookup
    table); the 15 decision thresholds are the midpoints of neighbouring table
    entries (exact in fp32)."""
    global _CODEBOOK
    if _CODEBOOK is None:
        c, _, _ = lloyd_max_normal()
        c16 = c.astype(np.float16).astype(np.float64)
        t = (c16[:-1] + c16[1:]) / 2.0
        _CODEBOOK = (c16.astype(np.float32), t.astype(np.float32))
    return _CODEBOOK


def tbq4_quantize(y: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Rotated fp32 blocks y [..., 128] -> (n16 float16 [...], indices uint8
    [..., 128]), with this op order (all fp32, round to nearest):

    * S = (p0 + p1) + (p2 + p3), p_k = the sum of y_i*y_i over the k-th run of
      32 values, accumulated in index order from 0;
    * n16 = fp16(min(sqrt(S), 65504)); nf = float(n16);
    * u_i = y_i / nf (0 when nf = 0); index_i = the number of thresholds
      strictly below u_i.
    """
    y = np.asarray(y, np.float32)
    _, thr = tbq4_codebook()
    sq = (y * y).astype(np.float32).reshape(*y.shape[:-1], 4, 32)
    p = np.zeros(sq.shape[:-1], np.float32)
    for e in range(32):
        p = (p + sq[..., e]).astype(np.float32)
    S = ((p[..., 0] + p[..., 1]).astype(np.float32) + (p[..., 2] + p[..., 3]).astype(np.float32)).astype(np.float32)
    n16 = np.minimum(np.sqrt(S).astype(np.float32), np.float32(65504.0)).astype(np.float16)
    nf = n16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        u = np.where(nf > 0, np.divide(y, nf, dtype=np.float32), np.float32(0.0))
    idx = (u[..., None] > thr).sum(axis=-1).astype(np.uint8)
    return n16, idx


def tbq4_quantize_f64norm(y: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """TBQ4 blocks with the norm read as its plain definition (trefon.com,
    "Jak 4-bitowemu cache to uchodzi: najpierw obrot": one fp16 L2 norm per
    block): n16 = fp16(min(sqrt(sum y_i^2), 65504)) with the sum and the root
    in fp64, then the same fp32 quotient and nearest-entry index as
    tbq4_quantize.  The format fixes no summation order; this variant shows
    how far the indices move when the order changes."""
    y = np.asarray(y, np.float32)
    _, thr = tbq4_codebook()
    S = np.sum(y.astype(np.float64) ** 2, axis=-1)
    n16 = np.minimum(np.sqrt(S), 65504.0).astype(np.float16)
    nf = n16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        u = np.where(nf > 0, np.divide(y, nf, dtype=np.float32), np.float32(0.0))
    idx = (u[..., None] > thr).sum(axis=-1).astype(np.uint8)
    return n16, idx


def tbq4_dequantize_f64(n16: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """table entry (an fp16 value) * norm, exact in fp64."""
    cent, _ = tbq4_codebook()
    return cent.astype(np.float64)[np.asarray(idx, np.int64)] * np.asarray(n16, np.float16).astype(np.float64)[..., None]


# ----------------------------------------------------------------------------
# Packing
# ----------------------------------------------------------------------------


def pack(codes: np.ndarray, bits: int) -> np.ndarray:
    """Pack int codes of the last axis (length G) into G*bits/8 bytes.

    8-bit: two's complement byte.  4-bit: nibble code+8, element 2i in the low
    nibble of byte i.  3-bit: code+4 in 3 bits, eight values per 24-bit
    little-endian word, value j at bits [3j, 3j+3).  2-bit: code+2, value j of
    a byte at bits [2j, 2j+2).
    """
    c = np.asarray(codes, np.int64)
    G = c.shape[-1]
    lead = c.shape[:-1]
    if bits == 8:
        return (c & 0xFF).astype(np.uint8)
    if bits == 4:
        u = (c + 8).reshape(*lead, G // 2, 2)
        return (u[..., 0] | (u[..., 1] << 4)).astype(np.uint8)
    if bits == 3:
        u = (c + 4).reshape(*lead, G // 8, 8)
        w = np.zeros(u.shape[:-1], np.int64)
        for j in range(8):
            w |= u[..., j] << (3 * j)
        out = np.stack([(w >> (8 * k)) & 0xFF for k in range(3)], axis=-1)
        return out.reshape(*lead, G // 8 * 3).astype(np.uint8)
    if bits == 2:
        u = (c + 2).reshape(*lead, G // 4, 4)
        b = u[..., 0] | (u[..., 1] << 2) | (u[..., 2] << 4) | (u[..., 3] << 6)
        return b.astype(np.uint8)
    raise ValueError(bits)


def unpack(payload: np.ndarray, bits: int, G: int) -> np.ndarray:
    """Inverse of pack: bytes [..., G*bits/8] -> int8 codes [..., G]."""
    p = np.asarray(payload, np.int64)
    lead = p.shape[:-1]
    if bits == 8:
        return np.where(p >= 128, p - 256, p).astype(np.int8)
    if bits == 4:
        lo = p & 0xF
        hi = (p >> 4) & 0xF
        return (np.stack([lo, hi], axis=-1).reshape(*lead, G) - 8).astype(np.int8)
    if bits == 3:
        t = p.reshape(*lead, G // 8, 3)
        w = t[..., 0] | (t[..., 1] << 8) | (t[..., 2] << 16)
        v = np.stack([(w >> (3 * j)) & 7 for j in range(8)], axis=-1)
        return (v.reshape(*lead, G) - 4).astype(np.int8)
    if bits == 2:
        v = np.stack([(p >> (2 * j)) & 3 for j in range(4)], axis=-1)
        return (v.reshape(*lead, G) - 2).astype(np.int8)
    raise ValueError(bits)


def encode_blocks(x: np.ndarray, bits: int, codebook: bool = False, zp: bool = False) -> np.ndarray:
    """fp32 blocks [..., G] -> bytes [..., block_bytes]: fp16 scale (little
    endian) then the packed codes.  codebook: TBQ4 blocks (the fp16 is the
    norm, the nibbles are centroid indices 0..15).  zp: asymmetric blocks
    (fp16 scale, fp16 zero, then the codes 0..2^b-1 in the same bit fields)."""
    if zp:
        s16, z16, c = quantize_zp(x, bits)
        sb = np.asarray(s16, np.float16).reshape(*s16.shape, 1).view(np.uint8)
        zb = np.asarray(z16, np.float16).reshape(*z16.shape, 1).view(np.uint8)
        return np.concatenate([sb, zb, pack(c.astype(np.int64) - _PACK_BIAS[bits], bits)], axis=-1)
    if codebook:
        s16, idx = tbq4_quantize(x)
        codes = idx.astype(np.int64) - 8
    else:
        s16, codes = quantize(x, bits)
    sb = np.asarray(s16, np.float16).reshape(*s16.shape, 1).view(np.uint8)
    return np.concatenate([sb, pack(codes, bits)], axis=-1)


def decode_blocks_zp(blob: np.ndarray, bits: int, G: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """asymmetric block bytes -> (s16, z16 float16 [...], codes uint8 [..., G])."""
    blob = np.ascontiguousarray(blob, np.uint8)
    s16 = blob[..., 0:2].copy().view(np.float16)[..., 0]
    z16 = blob[..., 2:4].copy().view(np.float16)[..., 0]
    codes = (unpack(blob[..., 4:], bits, G).astype(np.int64) + _PACK_BIAS[bits]).astype(np.uint8)
    return s16, z16, codes


def decode_blocks(blob: np.ndarray, bits: int, G: int) -> Tuple[np.ndarray, np.ndarray]:
    """bytes [..., block_bytes] -> (s16 float16 [...], codes int8 [..., G])."""
    blob = np.ascontiguousarray(blob, np.uint8)
    s16 = blob[..., 0:2].copy().view(np.float16)[..., 0]
    return s16, unpack(blob[..., 2:], bits, G)


# ----------------------------------------------------------------------------
# Cache buffers (byte layout described in the module docstring)
# ----------------------------------------------------------------------------


def row_bytes(fmt: Fmt, D: int) -> int:
    """Bytes of one storage row: a token row (per-token) or a group row (per-channel)."""
    bb = block_bytes(fmt.bits, fmt.group, fmt.zp)
    return (D // fmt.group) * bb if fmt.axis == AXIS_TOKEN else D * bb


def _tier_rows(cfg: Config, fmt: Fmt, ring: bool) -> int:
    if fmt.axis == AXIS_TOKEN:
        return (cfg.hot_window + unit_tokens(cfg)) if ring else -(-cfg.max_T // 32) * 32
    if ring:
        return cfg.hot_window // fmt.group + 1
    return -(-cfg.max_T // fmt.group)


def buffer_shapes(cfg: Config) -> Dict[str, Tuple[Tuple[int, ...], type]]:
    out = {}
    tiered = cfg.hot_window > 0
    for name, fmt in (("k_main", cfg.k_fmt), ("v_main", cfg.v_fmt)):
        rb = row_bytes(fmt, cfg.D)
        if cfg.page_tokens > 0:
            out[name] = ((cfg.L, cfg.n_pages, cfg.H_kv, cfg.page_tokens, rb), np.uint8)
        else:
            out[name] = ((cfg.L, cfg.batch, cfg.H_kv, _tier_rows(cfg, fmt, tiered), rb), np.uint8)
    if tiered:
        for name, fmt in (("k_cold", cfg.k_cold), ("v_cold", cfg.v_cold)):
            out[name] = ((cfg.L, cfg.batch, cfg.H_kv, _tier_rows(cfg, fmt, False), row_bytes(fmt, cfg.D)), np.uint8)
    rs = ring_slots(cfg)
    if rs:
        for name in ("k_resid", "v_resid"):
            out[name] = ((cfg.L, cfg.batch, cfg.H_kv, rs, cfg.D), np.uint16)
    return out


def new_buffers(cfg: Config) -> Dict[str, np.ndarray]:
    return {k: np.zeros(s, dt) for k, (s, dt) in buffer_shapes(cfg).items()}


def _main_token_row(cfg, bufs, name, layer, seq, h, t, block_table):
    """(array, index) of the per-token row of token t in the main tier."""
    if cfg.page_tokens > 0:
        page = int(block_table[seq, t // cfg.page_tokens])
        return bufs[name], (layer, page, h, t % cfg.page_tokens)
    if cfg.hot_window > 0:
        slots = cfg.hot_window + unit_tokens(cfg)
        return bufs[name], (layer, seq, h, t % slots)
    return bufs[name], (layer, seq, h, t)


def _main_group_row(cfg, name, layer, seq, h, gi):
    if cfg.hot_window > 0:
        fmt = cfg.k_fmt if name.startswith("k") else cfg.v_fmt
        return (layer, seq, h, gi % (cfg.hot_window // fmt.group + 1))
    return (layer, seq, h, gi)


# ----------------------------------------------------------------------------
# Append (quantize on write, window, tiers)
# ----------------------------------------------------------------------------


def _rotation_for(cfg: Config, which: str) -> bool:
    return bool(cfg.flags & (ROTATE_K if which == "k" else ROTATE_V))


def _codebook_for(cfg: Config, which: str) -> bool:
    return bool(cfg.flags & (TBQ4_K if which == "k" else TBQ4_V))


def quantize_rows(cfg: Config, fmt: Fmt, x: np.ndarray, rotate: bool, signs, codebook: bool = False) -> np.ndarray:
    """fp32 values [n_tok, H_kv, D] -> storage rows.

    Per-token: [n_tok, H_kv, row], each token on its own (rotated first when
    asked).  Per-channel: n_tok is a multiple of the group; returns
    [n_tok/G, H_kv, row], block c of a group row = channel c over the group's
    tokens in token order.
    """
    D = cfg.D
    if fmt.axis == AXIS_TOKEN:
        if rotate:
            x = rotate_f32(x, *signs)
        blocks = x.reshape(*x.shape[:-1], D // fmt.group, fmt.group)
        return encode_blocks(blocks, fmt.bits, codebook, fmt.zp).reshape(*x.shape[:-1], -1)
    G = fmt.group
    n_units = x.shape[0] // G
    xt = np.transpose(x.reshape(n_units, G, x.shape[1], D), (0, 2, 3, 1))  # [u, H, D, G]
    return encode_blocks(xt, fmt.bits, zp=fmt.zp).reshape(n_units, x.shape[1], -1)


def dequant_rows_f32(cfg: Config, fmt: Fmt, rows: np.ndarray) -> np.ndarray:
    """Storage rows -> fp32 values in the stored (possibly rotated) domain,
    [n_tok, H_kv, D]; the inverse of quantize_rows up to rounding."""
    D = cfg.D
    bb = block_bytes(fmt.bits, fmt.group, fmt.zp)
    def deq(blk):
        if fmt.zp:
            return dequantize_zp_f32(*decode_blocks_zp(blk, fmt.bits, fmt.group))
        return dequantize_f32(*decode_blocks(blk, fmt.bits, fmt.group))

    if fmt.axis == AXIS_TOKEN:
        blk = rows.reshape(*rows.shape[:-1], D // fmt.group, bb)
        return deq(blk).reshape(*rows.shape[:-1], D)
    n_units, H = rows.shape[0], rows.shape[1]
    v = deq(rows.reshape(n_units, H, D, bb))  # [u, H, D, G]
    return np.transpose(v, (0, 3, 1, 2)).reshape(n_units * fmt.group, H, D)


def _hot_index(cfg: Config, fmt: Fmt, seq: int, start: int, stop: int, block_table):
    """Index tuples (without the layer) of the main-tier rows holding tokens
    (per-token) or groups (per-channel) [start, stop)."""
    n = np.arange(start, stop)
    if cfg.page_tokens > 0:
        pages = np.asarray(block_table)[seq, n // cfg.page_tokens]
        return pages, n % cfg.page_tokens
    if cfg.hot_window > 0:
        if fmt.axis == AXIS_TOKEN:
            return seq, n % (cfg.hot_window + unit_tokens(cfg))
        return seq, n % (cfg.hot_window // fmt.group + 1)
    return seq, n


def _read_main(cfg, bufs, name, fmt, layer, seq, start, stop, block_table):
    """Main-tier rows [start, stop) (tokens or groups) as [n, H_kv, row]."""
    a, r = _hot_index(cfg, fmt, seq, start, stop, block_table)
    if cfg.page_tokens > 0:
        lay = bufs[name][layer]          # [pages, H, page_tokens, row]
        return lay[a, :, r]              # -> [n, H, row]
    blk = bufs[name][layer, a]           # [H, rows, row]
    return np.moveaxis(blk[:, r], 1, 0)  # -> [n, H, row]


def _write_main(cfg, bufs, name, fmt, layer, seq, start, stop, rows, block_table):
    """Store rows [n, H_kv, row] at main-tier positions [start, stop)."""
    a, r = _hot_index(cfg, fmt, seq, start, stop, block_table)
    if cfg.page_tokens > 0:
        lay = bufs[name][layer]
        lay[a, :, r] = rows
    else:
        blk = bufs[name][layer, a]
        blk[:, r] = np.moveaxis(rows, 0, 1)


def append(cfg: Config, bufs: Dict[str, np.ndarray], layer: int, k_new: np.ndarray,
           v_new: np.ndarray, n_new, seq_lens, block_table=None) -> None:
    """Append new tokens of one layer for every sequence, in place.

    k_new, v_new: uint16 raw input-dtype bits [total_new, H_kv, D], sequences
    back to back in batch order; n_new[b] new tokens of sequence b, whose cache
    holds seq_lens[b] tokens before the call.

    For each sequence, with T0 -> T1 the length before and after:
      (A) hot units [c_end(T0), min(c_end(T1), q_end(T0))) are requantized to
          the cold format from their dequantized hot values;
      (B) units [q_end(T0), q_end(T1)) are quantized from the window (tokens
          < T0) or the new input; a unit below c_end(T1) goes on to the cold
          format through the same hot quantize -> dequantize -> requantize;
      (C) new tokens in [max(T0, q_end(T1)), T1) are written to the window.
    """
    gam = unit_tokens(cfg)
    rs = ring_slots(cfg)
    signs = hadamard_signs(cfg.sign_seed)
    tiered = cfg.hot_window > 0
    off = 0
    for b in range(cfg.batch):
        n = int(n_new[b])
        T0 = int(seq_lens[b])
        T1 = T0 + n
        if T1 > cfg.max_T:
            raise ValueError("capacity")
        q0, q1 = q_end(cfg, T0), q_end(cfg, T1)
        c0, c1 = c_end(cfg, T0), c_end(cfg, T1)
        for which, new in (("k", k_new[off:off + n]), ("v", v_new[off:off + n])):
            fmt = cfg.k_fmt if which == "k" else cfg.v_fmt
            cold = (cfg.k_cold if which == "k" else cfg.v_cold) if tiered else None
            main = which + "_main"
            per_ch = fmt.axis == AXIS_CHANNEL

            def unit_range(t0, t1):
                return (t0 // gam, t1 // gam) if per_ch else (t0, t1)

            # (A) hot -> cold for units quantized before this call
            a0, a1 = c0, min(c1, q0)
            if a1 > a0:
                lo, hi = unit_range(a0, a1)
                rows = _read_main(cfg, bufs, main, fmt, layer, b, lo, hi, block_table)
                x = dequant_rows_f32(cfg, fmt, rows)
                bufs[which + "_cold"][layer, b, :, lo:hi] = np.moveaxis(
                    quantize_rows(cfg, cold, x, False, signs), 0, 1)
            # (B) newly quantized units
            if q1 > q0:
                t = np.arange(q0, q1)
                old = t < T0
                raw = np.empty((q1 - q0, cfg.H_kv, cfg.D), np.uint16)
                if old.any():
                    ring = bufs[which + "_resid"][layer, b]          # [H, slots, D]
                    raw[old] = np.moveaxis(ring[:, t[old] % rs], 1, 0)
                if (~old).any():
                    raw[~old] = new[t[~old] - T0]
                x = input_to_f32(raw, cfg.in_dtype)
                rows = quantize_rows(cfg, fmt, x, _rotation_for(cfg, which), signs, _codebook_for(cfg, which))
                split = min(max(c1, q0), q1) if tiered else q0  # units below `split` go cold
                ns = (split - q0) // gam if per_ch else split - q0
                if ns > 0:
                    xc = dequant_rows_f32(cfg, fmt, rows[:ns])
                    lo, hi = unit_range(q0, split)
                    bufs[which + "_cold"][layer, b, :, lo:hi] = np.moveaxis(
                        quantize_rows(cfg, cold, xc, False, signs), 0, 1)
                if split < q1:
                    lo, hi = unit_range(split, q1)
                    _write_main(cfg, bufs, main, fmt, layer, b, lo, hi, rows[ns:], block_table)
            # (C) window
            w0 = max(T0, q1)
            if T1 > w0:
                t = np.arange(w0, T1)
                ring = bufs[which + "_resid"][layer, b]
                ring[:, t % rs] = np.moveaxis(new[t - T0], 0, 1)
        off += n


# ----------------------------------------------------------------------------
# Dequantize and decode attention (fp64)
# ----------------------------------------------------------------------------


def dequantize(cfg: Config, bufs: Dict[str, np.ndarray], layer: int, seq: int, T: int,
               t0: int = 0, t1: Optional[int] = None, block_table=None,
               heads=None) -> Tuple[np.ndarray, np.ndarray]:
    """K, V of tokens [t0, t1) of one (layer, seq) as fp64 [n, H, D] in the
    original domain (rotation undone; keys as stored, pre-RoPE when stored so).
    x = code * scale is exact in fp64."""
    if t1 is None:
        t1 = T
    heads = np.arange(cfg.H_kv) if heads is None else np.asarray(heads)
    gam = unit_tokens(cfg)
    rs = ring_slots(cfg)
    qe, ce = q_end(cfg, T), c_end(cfg, T)
    signs = hadamard_signs(cfg.sign_seed)
    out = {}
    for which in ("k", "v"):
        fmt = cfg.k_fmt if which == "k" else cfg.v_fmt
        cold = cfg.k_cold if which == "k" else cfg.v_cold
        main = which + "_main"
        res = np.zeros((t1 - t0, len(heads), cfg.D), np.float64)
        for lo, hi, tier in ((0, ce, "cold"), (ce, qe, "main"), (qe, T, "window")):
            lo, hi = max(lo, t0), min(hi, t1)
            if hi <= lo:
                continue
            if tier == "window":
                t = np.arange(lo, hi)
                raw = bufs[which + "_resid"][layer, seq][np.ix_(heads, t % rs)]  # [H, n, D]
                res[lo - t0:hi - t0] = np.moveaxis(input_to_f32(raw, cfg.in_dtype), 0, 1)
                continue
            f = cold if tier == "cold" else fmt
            if f.axis == AXIS_CHANNEL:
                g_lo, g_hi = lo // gam, (hi + gam - 1) // gam
                if tier == "cold":
                    rows = np.moveaxis(bufs[which + "_cold"][layer, seq, :, g_lo:g_hi], 1, 0)
                else:
                    rows = _read_main(cfg, bufs, main, f, layer, seq, g_lo, g_hi, block_table)
                bb = block_bytes(f.bits, f.group, f.zp)
                rows = rows[:, heads]
                blk = rows.reshape(g_hi - g_lo, len(heads), cfg.D, bb)
                if f.zp:
                    v = dequantize_zp_f64(*decode_blocks_zp(blk, f.bits, f.group))  # [u, H, D, G]
                else:
                    s16, codes = decode_blocks(blk, f.bits, f.group)
                    v = codes.astype(np.float64) * s16.astype(np.float64)[..., None]  # [u, H, D, G]
                v = np.transpose(v, (0, 3, 1, 2)).reshape((g_hi - g_lo) * gam, len(heads), cfg.D)
                res[lo - t0:hi - t0] = v[lo - g_lo * gam:hi - g_lo * gam]
            else:
                if tier == "cold":
                    rows = np.moveaxis(bufs[which + "_cold"][layer, seq, :, lo:hi], 1, 0)
                else:
                    rows = _read_main(cfg, bufs, main, f, layer, seq, lo, hi, block_table)
                rows = rows[:, heads]
                bb = block_bytes(f.bits, f.group, f.zp)
                blk = rows.reshape(hi - lo, len(heads), cfg.D // f.group, bb)
                if f.zp:
                    s16, z16, zc = decode_blocks_zp(blk, f.bits, f.group)
                    codes = None
                else:
                    s16, codes = decode_blocks(blk, f.bits, f.group)
                if f.zp:
                    val = dequantize_zp_f64(s16, z16, zc).reshape(hi - lo, len(heads), cfg.D)
                elif _codebook_for(cfg, which):
                    val = tbq4_dequantize_f64(s16, codes.astype(np.int64) + 8).reshape(hi - lo, len(heads), cfg.D)
                else:
                    val = dequantize_f64(s16, codes).reshape(hi - lo, len(heads), cfg.D)
                if _rotation_for(cfg, which):
                    val = unrotate_f64(val, *signs)
                res[lo - t0:hi - t0] = val
        out[which] = res
    return out["k"], out["v"]


def rope_f64(k: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Split-half RoPE in fp64: pairs (i, i + D/2), angle t * theta^(-2i/D):
    k'_i = k_i cos - k_{i+D/2} sin, k'_{i+D/2} = k_i sin + k_{i+D/2} cos."""
    k = np.asarray(k, np.float64)
    D = k.shape[-1]
    h = D // 2
    inv = theta ** (-2.0 * np.arange(h, dtype=np.float64) / D)
    ang = np.asarray(positions, np.float64).reshape(-1, *([1] * (k.ndim - 1))) * inv
    c, s = np.cos(ang), np.sin(ang)
    a, b = k[..., :h], k[..., h:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def softmax_f64(s: np.ndarray) -> np.ndarray:
    m = np.max(s)
    e = np.exp(s - m)
    return e / np.sum(e)


def attention_f64(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """One head: s_i = q.k_i / sqrt(D); p = softmax(s); out = sum_i p_i v_i.
    An empty cache gives 0."""
    q = np.asarray(q, np.float64)
    if K.shape[0] == 0:
        return np.zeros(q.shape[-1], np.float64)
    s = (np.asarray(K, np.float64) @ q) / math.sqrt(q.shape[-1])
    p = softmax_f64(s)
    return p @ np.asarray(V, np.float64)


def scores_f64(q: np.ndarray, K: np.ndarray) -> np.ndarray:
    return (np.asarray(K, np.float64) @ np.asarray(q, np.float64)) / math.sqrt(q.shape[-1])


def decode_attention(cfg: Config, bufs: Dict[str, np.ndarray], layer0: int, n_layers: int,
                     q: np.ndarray, seq_lens, block_table=None, which=None) -> np.ndarray:
    """fp64 decode attention over the dequantized cache.

    q: raw input-dtype bits [n_layers, batch, H_q, D] (post-RoPE queries).
    which: optional list of (layer_offset, seq, q_head) to compute; others stay 0.
    Returns fp64 [n_layers, batch, H_q, D].
    """
    g = cfg.H_q // cfg.H_kv
    out = np.zeros((n_layers, cfg.batch, cfg.H_q, cfg.D), np.float64)
    wanted = None if which is None else set(which)
    for li in range(n_layers):
        for b in range(cfg.batch):
            heads_needed = [h for h in range(cfg.H_q) if wanted is None or (li, b, h) in wanted]
            if not heads_needed:
                continue
            T = int(seq_lens[b])
            kv_needed = sorted({h // g for h in heads_needed})
            K, V = dequantize(cfg, bufs, layer0 + li, b, T, block_table=block_table, heads=kv_needed)
            if cfg.flags & K_PRE_ROPE:
                K = rope_f64(K, np.arange(T), cfg.rope_theta)
            qf = input_to_f32(q[li, b], cfg.in_dtype).astype(np.float64)
            for h in heads_needed:
                j = kv_needed.index(h // g)
                out[li, b, h] = attention_f64(qf[h], K[:, j], V[:, j])
    return out
