// Kernels of the specialized phase B of quantize-on-append: 32-value blocks
// of unrotated formats.  Every translation unit that includes this header is
// compiled with --fmad=false like the generic kernels; each instantiates the
// kernels of the formats it launches.
#pragma once
#include "append_common.cuh"

namespace kvq {
namespace {

// ---- specialized phase B: 32-value blocks of unrotated formats ------------------
//
// Formats with 32-value blocks and no rotation get their own kernels, one per
// tensor (K or V), specialized on the bit width, the input dtype and the cold
// tier's bit width.  The inputs are 16-bit floats, so x / s16 is computed
// exactly without a divide: with rcp = RN(1/s), q0 = RN(x rcp) and the exact
// remainder e = x - q0 s (one fma), RN(q0 + e rcp) is RN(x / s) (Markstein's
// correction step, P. Markstein, IBM J. Res. Dev. 34(1), 1990).  Adding
// 1.5 * 2^23 (+ the storage bias) then rounds to the nearest integer, ties to
// even, like rint, and leaves the biased code in the low mantissa bits.  A
// block only needs the clamp to [-qmax, qmax] when its scale is subnormal or
// saturated in fp16 (otherwise |x / s16| <= qmax (1 + 2^-10) < qmax + 1/2);
// it is then applied to x, as |x| <= qmax s16 (an exact product), which
// gives the same codes as clamping the rounded quotient.

constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23
constexpr float kMinNormalF16 = 6.103515625e-05f;

template <int DT>
__device__ __forceinline__ float2 raw_pair_to_f32(uint32_t w) {
  if constexpr (DT == KVQ_DT_F16) {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
  } else {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  }
}

template <int DT>
__device__ __forceinline__ float in_to_f32_t(uint32_t bits16) {
  if constexpr (DT == KVQ_DT_F16) return __half2float(__ushort_as_half((unsigned short)bits16));
  else return __uint_as_float(bits16 << 16);
}

__device__ __forceinline__ float div_by_scale(float x, float sf, float rcp) {
  const float q0 = __fmul_rn(x, rcp);
  const float e = __fmaf_rn(-q0, sf, x);
  return __fmaf_rn(e, rcp, q0);
}

// Codes of v[0..31] with scale sf (rcp = RN(1/sf), 0 when sf = 0) as a
// 32*B-bit little-endian stream (biased codes; two's complement for B = 8);
// dq (optional) receives code * sf.  The rounded value's float bits are
// kRoundMagicBits + code + bias; each word accumulates those bits shifted into
// place (one integer multiply-add per code) and subtracts the magic parts
// once, which is exact modulo 2^32 because every biased code fits its field.
// For B = 8 the bias is 128 and flipping each byte's top bit afterwards gives
// two's complement.
constexpr uint32_t kRoundMagicBits = 0x4B400000u;  // bits of 1.5 * 2^23

template <int B>
__device__ __forceinline__ void codes32(const float (&v)[32], float sf, float rcp, uint32_t (&w)[B], float* dq) {
  constexpr int qmax = (1 << (B - 1)) - 1;
  constexpr int bias = qmax + 1;
  constexpr float magic = kRoundMagic + (float)bias;
  // the quotient and the rounding on pairs of values (each half rounded like
  // the scalar operation): q0 = RN(x rcp), e = RN(x - q0 s) exactly, RN(q0 + e rcp)
  const uint64_t R2 = pk2(rcp, rcp), NS2 = pk2(-sf, -sf), M2 = pk2(magic, magic);
#pragma unroll
  for (int k = 0; k < B; ++k) w[k] = 0;
  uint32_t corr[B];
#pragma unroll
  for (int k = 0; k < B; ++k) corr[k] = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint64_t X = pk2(v[2 * i], v[2 * i + 1]);
    const uint64_t Q0 = mul2(X, R2);
    const uint64_t Q1 = fma2(fma2(Q0, NS2, X), R2, Q0);
    const uint64_t R = add2(Q1, M2);
    float rr[2];
    upk2(R, rr[0], rr[1]);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int j = 2 * i + c;
      if (dq) dq[j] = __fmul_rn(__fsub_rn(rr[c], magic), sf);
      const uint32_t bits = __float_as_uint(rr[c]);
      const int bit = B * j, k = bit / 32, sh = bit % 32;
      if (sh + B > 32) {  // a 3-bit code across two words: place the true biased code
        const uint32_t u = bits - kRoundMagicBits;
        w[k] += u << sh;
        w[k + 1] += u >> (32 - sh);
      } else {
        w[k] += bits << sh;
        corr[k] += kRoundMagicBits << sh;
      }
    }
  }
#pragma unroll
  for (int k = 0; k < B; ++k) {
    w[k] -= corr[k];
    if (B == 8) w[k] ^= 0x80808080u;
  }
}

// One block of 32 values: scale of absolute maximum m, codes; the block (fp16
// scale then payload) goes to dst (2-byte aligned) when given.
template <int B>
__device__ __forceinline__ void block32(float (&v)[32], float m, uint8_t* dst, float* dq) {
  constexpr int qmax = (1 << (B - 1)) - 1;
  const __half s16 = block_scale_of(m, qmax);
  const float sf = __half2float(s16);
  const float rcp = sf == 0.f ? 0.f : __frcp_rn(sf);
  if (!(sf >= kMinNormalF16 && sf < 65504.f)) {
    const float lim = __fmul_rn((float)qmax, sf);
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = fminf(fmaxf(v[j], -lim), lim);
  }
  uint32_t w[B];
  codes32<B>(v, sf, rcp, w, dq);
  if (!dst) return;
  uint16_t* p = reinterpret_cast<uint16_t*>(dst);
  p[0] = __half_as_ushort(s16);
#pragma unroll
  for (int k = 0; k < B; ++k) {
    p[1 + 2 * k] = (uint16_t)w[k];
    p[2 + 2 * k] = (uint16_t)(w[k] >> 16);
  }
}

// Asymmetric block of 32 values (fp16 scale, fp16 zero, codes 0..2^B-1), in
// the format's op order: with mn, mx the block's minimum (a zero as +0) and
// maximum, s16 = fp16(min((mx - mn) / (2^B - 1), 65504)), z16 = fp16(mn
// clipped to +-65504), code = clamp(rint((x - z) / s), 0, 2^B - 1), 0 when
// s = 0.  The quotient RN(d / s) of d = RN(x - z) is taken with Markstein's
// correction step (as div_by_scale); with rcp = 0 when s = 0 it gives 0.
// The code is a nondecreasing function of x, so when the codes of the
// block's minimum and maximum lie in [0, 2^B - 1] no value needs the clamp;
// any other block (a saturated or nearly degenerate scale, an infinity) is
// quantized by the serial form, quant_zp32, with the IEEE divide and the clamp.
__device__ __forceinline__ float zp_magic_code(float x, float sf, float zf, float rcp) {
  return __fadd_rn(div_by_scale(__fsub_rn(x, zf), sf, rcp), kRoundMagic);
}

template <int B>
__device__ __forceinline__ void codes_zp(const float (&v)[32], float sf, float zf, float rcp, uint32_t (&w)[B],
                                         float* dq) {
  uint32_t corr[B];
#pragma unroll
  for (int k = 0; k < B; ++k) w[k] = corr[k] = 0;
  // x - z, the quotient and the rounding on pairs of values (each half
  // rounded like the scalar operation)
  const uint64_t Z2 = pk2(zf, zf), R2 = pk2(rcp, rcp), NS2 = pk2(-sf, -sf), M2 = pk2(kRoundMagic, kRoundMagic);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint64_t Dd = sub2(pk2(v[2 * i], v[2 * i + 1]), Z2);
    const uint64_t Q0 = mul2(Dd, R2);
    const uint64_t R0 = add2(fma2(fma2(Q0, NS2, Dd), R2, Q0), M2);
    float r0[2];
    upk2(R0, r0[0], r0[1]);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int j = 2 * i + c;
      const float r = r0[c];
      if (dq) dq[j] = __fadd_rn(__fmul_rn(__fsub_rn(r, kRoundMagic), sf), zf);
      const int bit = B * j, k = bit / 32, sh = bit % 32;
      w[k] += __float_as_uint(r) << sh;
      corr[k] += kRoundMagicBits << sh;
    }
  }
#pragma unroll
  for (int k = 0; k < B; ++k) w[k] -= corr[k];
}

template <int B>
__device__ __forceinline__ void block32_zp(const float (&v)[32], float mn, float mx, uint8_t* dst, float* dq) {
  constexpr int qlev = (1 << B) - 1;
  mn = __fadd_rn(mn, 0.0f);
  const __half s16 = __float2half_rn(fminf(__fdiv_rn(__fsub_rn(mx, mn), (float)qlev), 65504.0f));
  const __half z16 = __float2half_rn(fminf(fmaxf(mn, -65504.0f), 65504.0f));
  const float sf = __half2float(s16), zf = __half2float(z16);
  const float rcp = sf == 0.f ? 0.f : __frcp_rn(sf);
  if (!(zp_magic_code(mn, sf, zf, rcp) >= kRoundMagic &&
        zp_magic_code(mx, sf, zf, rcp) <= kRoundMagic + (float)qlev)) {
    quant_zp32(v, B, dst, dq);
    return;
  }
  uint32_t w[B];
  codes_zp<B>(v, sf, zf, rcp, w, dq);
  if (!dst) return;
  uint16_t* p = reinterpret_cast<uint16_t*>(dst);
  p[0] = __half_as_ushort(s16);
  p[1] = __half_as_ushort(z16);
#pragma unroll
  for (int k = 0; k < B; ++k) {
    p[2 + 2 * k] = (uint16_t)w[k];
    p[3 + 2 * k] = (uint16_t)(w[k] >> 16);
  }
}

__device__ __forceinline__ void minmax_of(const float (&v)[32], float& mn, float& mx) {
  mn = mx = v[0];
#pragma unroll
  for (int j = 1; j < 32; ++j) {
    mn = fminf(mn, v[j]);
    mx = fmaxf(mx, v[j]);
  }
}

// Elementwise min / max of two pairs of 16-bit floats (NaN-ignoring, like
// fminf / fmaxf; exact, so the fp32 extremes are those of the pairs).
template <int DT>
__device__ __forceinline__ uint32_t min2_16(uint32_t a, uint32_t b) {
  uint32_t d;
  if constexpr (DT == KVQ_DT_F16) asm("min.f16x2 %0, %1, %2;\n" : "=r"(d) : "r"(a), "r"(b));
  else asm("min.bf16x2 %0, %1, %2;\n" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
template <int DT>
__device__ __forceinline__ uint32_t max2_16(uint32_t a, uint32_t b) {
  uint32_t d;
  if constexpr (DT == KVQ_DT_F16) asm("max.f16x2 %0, %1, %2;\n" : "=r"(d) : "r"(a), "r"(b));
  else asm("max.bf16x2 %0, %1, %2;\n" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ float amax_of(const float (&v)[32]) {
  float m = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) m = fmaxf(m, fabsf(v[j]));
  return m;
}

// Hot block of v into dst, or (to_cold) the cold block of its dequantized
// values into dstc.  Z: asymmetric blocks in both tiers.
template <int B, int CB, bool Z = false>
__device__ __forceinline__ void hot_or_cold(float (&v)[32], bool to_cold, uint8_t* dst, uint8_t* dstc,
                                            float mn = 0.f, float mx = 0.f) {
  if constexpr (Z) {  // mn, mx: the block's minimum and maximum
    if constexpr (CB != 0) {
      if (to_cold) {
        float dq[32], cmn, cmx;
        block32_zp<B>(v, mn, mx, nullptr, dq);
        minmax_of(dq, cmn, cmx);
        block32_zp<CB>(dq, cmn, cmx, dstc, nullptr);
        return;
      }
    }
    block32_zp<B>(v, mn, mx, dst, nullptr);
    return;
  }
  if constexpr (CB != 0) {
    if (to_cold) {
      float dq[32];
      block32<B>(v, amax_of(v), nullptr, dq);
      block32<CB>(dq, amax_of(dq), dstc, nullptr);
      return;
    }
  }
  block32<B>(v, amax_of(v), dst, nullptr);
}

// Copies `bytes` (a multiple of 4) from shared `src` to global `dst` (4-byte
// aligned) with all threads of the block; 16-byte words when both allow.
__device__ __forceinline__ void block_copy_out(uint8_t* dst, const uint8_t* src, int bytes) {
  if (((reinterpret_cast<uintptr_t>(dst) | (uintptr_t)bytes) & 15u) == 0) {
    for (int e = threadIdx.x; e < bytes / 16; e += blockDim.x)
      reinterpret_cast<uint4*>(dst)[e] = reinterpret_cast<const uint4*>(src)[e];
  } else {
    for (int e = threadIdx.x; e < bytes / 4; e += blockDim.x)
      reinterpret_cast<uint32_t*>(dst)[e] = reinterpret_cast<const uint32_t*>(src)[e];
  }
}

// Two symmetric blocks at once: channels c and c + 1 of 32 tokens, raw[j]
// holding token j's two 16-bit values, each block as block32 computes it
// (absolute maxima on the 16-bit pairs, exact; the quotient, correction and
// rounding on f32x2 lanes, one per channel).  Returns false, writing
// nothing, when either scale is subnormal or saturated in fp16: those blocks
// need the clamp and go through block32 one by one.
template <int DT, int B>
__device__ __forceinline__ bool block32_x2(const uint32_t (&raw)[32], uint8_t* dst0, uint8_t* dst1) {
  constexpr int qmax = (1 << (B - 1)) - 1;
  constexpr float magic = kRoundMagic + (float)(qmax + 1);
  uint32_t a2 = raw[0] & 0x7FFF7FFFu;
#pragma unroll
  for (int j = 1; j < 32; ++j) a2 = max2_16<DT>(a2, raw[j] & 0x7FFF7FFFu);
  const float2 m = raw_pair_to_f32<DT>(a2);
  const __half s0 = block_scale_of(m.x, qmax), s1 = block_scale_of(m.y, qmax);
  const float f0 = __half2float(s0), f1 = __half2float(s1);
  if (!(f0 >= kMinNormalF16 && f0 < 65504.f && f1 >= kMinNormalF16 && f1 < 65504.f)) return false;
  const uint64_t R2 = pk2(__frcp_rn(f0), __frcp_rn(f1)), NS2 = pk2(-f0, -f1), M2 = pk2(magic, magic);
  uint32_t w0[B], w1[B], corr[B];
#pragma unroll
  for (int k = 0; k < B; ++k) w0[k] = w1[k] = corr[k] = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float2 x = raw_pair_to_f32<DT>(raw[j]);
    const uint64_t X = pk2(x.x, x.y);
    const uint64_t Q0 = mul2(X, R2);
    float r0, r1;
    upk2(add2(fma2(fma2(Q0, NS2, X), R2, Q0), M2), r0, r1);
    const uint32_t b0 = __float_as_uint(r0), b1 = __float_as_uint(r1);
    const int bit = B * j, k = bit / 32, sh = bit % 32;
    if (sh + B > 32) {  // a 3-bit code across two words: place the true biased code
      const uint32_t u0 = b0 - kRoundMagicBits, u1 = b1 - kRoundMagicBits;
      w0[k] += u0 << sh;
      w0[k + 1] += u0 >> (32 - sh);
      w1[k] += u1 << sh;
      w1[k + 1] += u1 >> (32 - sh);
    } else {
      w0[k] += b0 << sh;
      w1[k] += b1 << sh;
      corr[k] += kRoundMagicBits << sh;
    }
  }
  uint16_t* p0 = reinterpret_cast<uint16_t*>(dst0);
  uint16_t* p1 = reinterpret_cast<uint16_t*>(dst1);
  p0[0] = __half_as_ushort(s0);
  p1[0] = __half_as_ushort(s1);
#pragma unroll
  for (int k = 0; k < B; ++k) {
    uint32_t a = w0[k] - corr[k], b = w1[k] - corr[k];
    if (B == 8) {
      a ^= 0x80808080u;
      b ^= 0x80808080u;
    }
    p0[1 + 2 * k] = (uint16_t)a;
    p0[2 + 2 * k] = (uint16_t)(a >> 16);
    p1[1 + 2 * k] = (uint16_t)b;
    p1[2 + 2 * k] = (uint16_t)(b >> 16);
  }
  return true;
}

// The blocks block32_x2 declines (a subnormal or saturated scale), one
// channel at a time through block32; out of line, with the 16-bit pairs in
// local memory, so that the common path keeps its registers.
template <int DT, int B>
__device__ __noinline__ void block32_pair_slow(const uint32_t* raw, uint8_t* dst0, uint8_t* dst1) {
  for (int hc = 0; hc < 2; ++hc) {
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = in_to_f32_t<DT>(hc ? (raw[j] >> 16) : (raw[j] & 0xFFFFu));
    block32<B>(v, amax_of(v), hc ? dst1 : dst0, nullptr);
  }
}

// Cold 2-bit blocks straight from 16-bit inputs.  A token that enters the
// cache in the cold tier is quantized to its hot block, dequantized and
// quantized again to 2 bits (the tiers' op order).  For a symmetric hot block
// with a normal fp16 scale s = fp16(amax / qmax), amax / s lies within
// qmax 2^-10 of qmax, so the largest hot code magnitude is qmax (odd), the
// cold block's absolute maximum is qmax s (exact in fp32) and its scale is
// c = fp16(qmax s), within 2^-11 of qmax s.  A hot magnitude m then gets the
// cold magnitude rint(m s / c): m s / c lies within 2^-10 of m / qmax, which is
// at least 1/2 + 1/(2 qmax) for m >= k = (qmax + 1) / 2 = 2^(B-2) and at most
// 1/2 - 1/(2 qmax) below it, so the cold code is nonzero exactly when m >= k.
// m = rint(q) for the fp32 quotient q = RN(|x| / s) reaches k when
// q >= k - 1/2 (a tie rounds to k when k is even, B >= 3) or q > k - 1/2
// (k = 1, B = 2); and since a 16-bit x over an fp16 s never has an fp32
// quotient that rounds onto k - 1/2 from either side, that is |x| >= th
// (or > th) for th = (k - 1/2) s, an exact fp32 product.  In 16-bit terms:
// |x| >= ru16(th) (or |x| > rd16(th)), one packed compare per pair of values.
// The cold code is sign(x) where nonzero.  Blocks whose hot scale is
// subnormal or saturated, or whose cold scale saturates, go the two-pass way.
template <int DT, int B>
__device__ __forceinline__ bool cold2_rule(float amax, uint16_t& thr, __half& c16) {
  static_assert(B >= 2 && B <= 8, "hot bits");
  constexpr int qmax = (1 << (B - 1)) - 1;
  const float sf = __half2float(block_scale_of(amax, qmax));
  if (!(sf >= kMinNormalF16 && sf < 65504.f)) return false;
  c16 = __float2half_rn(__fmul_rn((float)qmax, sf));  // the cold block's scale, qmax s / 1
  if (!(__half2float(c16) < 65504.f)) return false;
  const float th = __fmul_rn((float)(1 << (B - 2)) - 0.5f, sf);
  if constexpr (DT == KVQ_DT_F16)
    thr = __half_as_ushort(B >= 3 ? __float2half_ru(th) : __float2half_rd(th));
  else
    thr = __bfloat16_as_ushort(B >= 3 ? __float2bfloat16_ru(th) : __float2bfloat16_rd(th));
  return true;
}

// Per half of x: 0xFFFF when |x| passes the threshold t (>= for B >= 3, >
// for B = 2), else 0.
template <int DT, int B>
__device__ __forceinline__ uint32_t cold2_mask(uint32_t x, uint32_t t) {
  if constexpr (DT == KVQ_DT_F16) {
    const __half2 a = __habs2(*reinterpret_cast<const __half2*>(&x)), b = *reinterpret_cast<const __half2*>(&t);
    return B >= 3 ? __hge2_mask(a, b) : __hgt2_mask(a, b);
  } else {
    const __nv_bfloat162 a = __habs2(*reinterpret_cast<const __nv_bfloat162*>(&x));
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&t);
    return B >= 3 ? __hge2_mask(a, b) : __hgt2_mask(a, b);
  }
}

// The 2-bit fields of eight pairs p[0..7]: pair e's low value at bits 2e,
// its high value at bits 16 + 2e, each field (nonzero, nonzero and negative)
// so that field ^ 2 is the biased cold code (1, 2, 3 for -1, 0, +1).  Each
// pair's fields enter at bits 14 and 30 and move down two bits per later pair.
template <int DT, int B>
__device__ __forceinline__ uint32_t cold2_fields8(const uint32_t* p, uint32_t thr2) {
  uint32_t q = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const uint32_t m = cold2_mask<DT, B>(p[e], thr2);
    q = (q >> 2) | (m & (p[e] | 0x40004000u) & 0xC000C000u);
  }
  return q;
}

// 2-bit fields L0..L7 (low half) and H0..H7 (high half) of x as L0 H0 L1 H1 ...
__device__ __forceinline__ uint32_t interleave2(uint32_t x) {
  x = __byte_perm(x, 0, 0x3120);
  x = (x & 0xF00FF00Fu) | ((x & 0x00F000F0u) << 4) | ((x >> 4) & 0x00F000F0u);
  return (x & 0xC3C3C3C3u) | ((x & 0x0C0C0C0Cu) << 2) | ((x >> 2) & 0x0C0C0C0Cu);
}

__device__ __forceinline__ void put_cold2(uint8_t* dst, __half c16, uint32_t w0, uint32_t w1) {
  uint16_t* p = reinterpret_cast<uint16_t*>(dst);
  w0 ^= 0xAAAAAAAAu;
  w1 ^= 0xAAAAAAAAu;
  p[0] = __half_as_ushort(c16);
  p[1] = (uint16_t)w0;
  p[2] = (uint16_t)(w0 >> 16);
  p[3] = (uint16_t)w1;
  p[4] = (uint16_t)(w1 >> 16);
}

// One cold block from a 32-value slice of a token row (w[e] holding values
// 2e and 2e + 1).  Returns false, writing nothing, where the rule above does
// not apply.
template <int DT, int B>
__device__ __forceinline__ bool cold2_slice(const uint32_t (&w)[16], uint8_t* dst) {
  uint32_t a2 = w[0] & 0x7FFF7FFFu;
#pragma unroll
  for (int e = 1; e < 16; ++e) a2 = max2_16<DT>(a2, w[e] & 0x7FFF7FFFu);
  const float2 m = raw_pair_to_f32<DT>(a2);
  uint16_t thr;
  __half c16;
  if (!cold2_rule<DT, B>(fmaxf(m.x, m.y), thr, c16)) return false;
  const uint32_t t2 = thr * 0x00010001u;
  put_cold2(dst, c16, interleave2(cold2_fields8<DT, B>(w, t2)), interleave2(cold2_fields8<DT, B>(w + 8, t2)));
  return true;
}

// Two cold blocks: channels c and c + 1 of 32 tokens, raw[j] holding token
// j's two 16-bit values.  Returns false, writing nothing, where the rule
// above does not apply to either block.
template <int DT, int B>
__device__ __forceinline__ bool cold2_x2(const uint32_t (&raw)[32], uint8_t* dst0, uint8_t* dst1) {
  uint32_t a2 = raw[0] & 0x7FFF7FFFu;
#pragma unroll
  for (int j = 1; j < 32; ++j) a2 = max2_16<DT>(a2, raw[j] & 0x7FFF7FFFu);
  const float2 m = raw_pair_to_f32<DT>(a2);
  uint16_t t0, t1;
  __half c0, c1;
  if (!(cold2_rule<DT, B>(m.x, t0, c0) && cold2_rule<DT, B>(m.y, t1, c1))) return false;
  const uint32_t t2 = t0 | ((uint32_t)t1 << 16);
  uint32_t q[4];
#pragma unroll
  for (int g = 0; g < 4; ++g) q[g] = cold2_fields8<DT, B>(raw + 8 * g, t2);
  put_cold2(dst0, c0, __byte_perm(q[0], q[1], 0x5410), __byte_perm(q[2], q[3], 0x5410));
  put_cold2(dst1, c1, __byte_perm(q[0], q[1], 0x7632), __byte_perm(q[2], q[3], 0x7632));
  return true;
}

// The blocks the direct rule declines, one channel at a time the two-pass
// way; out of line, with the 16-bit pairs in local memory.
template <int DT, int B, int CB>
__device__ __noinline__ void cold_pair_slow(const uint32_t* raw, uint8_t* dst0, uint8_t* dst1) {
  for (int hc = 0; hc < 2; ++hc) {
    float v[32], dq[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = in_to_f32_t<DT>(hc ? (raw[j] >> 16) : (raw[j] & 0xFFFFu));
    block32<B>(v, amax_of(v), nullptr, dq);
    block32<CB>(dq, amax_of(dq), hc ? dst1 : dst0, nullptr);
  }
}

// Two asymmetric blocks at once: channels c and c + 1 of 32 tokens, raw[j]
// holding token j's two 16-bit values.  The codes of both blocks are taken on
// f32x2 pairs (one lane per channel) as codes_zp does, consuming raw as they
// go; when either block needs the clamp, both go through the serial form.
template <int DT, int B>
__device__ __forceinline__ void block32_zp_x2(const uint32_t (&raw)[32], float2 mn, float2 mx, uint8_t* dst0,
                                              uint8_t* dst1) {
  constexpr int qlev = (1 << B) - 1;
  float sf[2], zf[2], rcp[2];
  __half s16[2], z16[2];
  bool ok = true;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const float lo = __fadd_rn(c ? mn.y : mn.x, 0.0f), hi = c ? mx.y : mx.x;
    s16[c] = __float2half_rn(fminf(__fdiv_rn(__fsub_rn(hi, lo), (float)qlev), 65504.0f));
    z16[c] = __float2half_rn(fminf(fmaxf(lo, -65504.0f), 65504.0f));
    sf[c] = __half2float(s16[c]);
    zf[c] = __half2float(z16[c]);
    rcp[c] = sf[c] == 0.f ? 0.f : __frcp_rn(sf[c]);
    ok = ok && zp_magic_code(lo, sf[c], zf[c], rcp[c]) >= kRoundMagic &&
         zp_magic_code(hi, sf[c], zf[c], rcp[c]) <= kRoundMagic + (float)qlev;
  }
  if (!ok) {
#pragma unroll 1
    for (int c = 0; c < 2; ++c) {
      float t[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) t[j] = in_to_f32_t<DT>(c ? (raw[j] >> 16) : (raw[j] & 0xFFFFu));
      quant_zp32_mem(t, B, c ? dst1 : dst0, nullptr);
    }
    return;
  }
  const uint64_t Z2 = pk2(zf[0], zf[1]), R2 = pk2(rcp[0], rcp[1]), NS2 = pk2(-sf[0], -sf[1]),
                 M2 = pk2(kRoundMagic, kRoundMagic);
  uint32_t w0[B], w1[B], corr[B];
#pragma unroll
  for (int k = 0; k < B; ++k) w0[k] = w1[k] = corr[k] = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float2 x = raw_pair_to_f32<DT>(raw[j]);
    const uint64_t Dd = sub2(pk2(x.x, x.y), Z2);
    const uint64_t Q0 = mul2(Dd, R2);
    float r0, r1;
    upk2(add2(fma2(fma2(Q0, NS2, Dd), R2, Q0), M2), r0, r1);
    const int bit = B * j, k = bit / 32, sh = bit % 32;
    w0[k] += __float_as_uint(r0) << sh;
    w1[k] += __float_as_uint(r1) << sh;
    corr[k] += kRoundMagicBits << sh;
  }
  uint16_t* p0 = reinterpret_cast<uint16_t*>(dst0);
  uint16_t* p1 = reinterpret_cast<uint16_t*>(dst1);
  p0[0] = __half_as_ushort(s16[0]);
  p0[1] = __half_as_ushort(z16[0]);
  p1[0] = __half_as_ushort(s16[1]);
  p1[1] = __half_as_ushort(z16[1]);
#pragma unroll
  for (int k = 0; k < B; ++k) {
    const uint32_t a = w0[k] - corr[k], b = w1[k] - corr[k];
    p0[2 + 2 * k] = (uint16_t)a;
    p0[3 + 2 * k] = (uint16_t)(a >> 16);
    p1[2 + 2 * k] = (uint16_t)b;
    p1[3 + 2 * k] = (uint16_t)(b >> 16);
  }
}

// Rows [r0, r1) of a shared tile of W-word rows (row r at src + 4 W r) to
// their destinations d[r], skipping null ones: word e of the run goes to
// thread e mod blockDim.x.
template <int W>
__device__ __forceinline__ void rows_out(uint8_t* const* d, const uint8_t* src, int r0, int r1) {
  const uint32_t* s = reinterpret_cast<const uint32_t*>(src);
  for (int e = r0 * W + (int)threadIdx.x; e < r1 * W; e += blockDim.x) {
    const int r = e / W;
    uint32_t* row = reinterpret_cast<uint32_t*>(d[r]);
    if (row) row[e - r * W] = s[e];
  }
}

// Per-token 32-value blocks: a block of 128 threads takes 128 consecutive
// tokens of one (layer, sequence, kv head); thread j quantizes token row j
// slice by slice.  At D = 128 (when the static shared memory allows) the rows
// arrive through a shared stage filled by cp.async with 16 consecutive threads
// per 256-byte row: a load of each thread's own row touches 32 lines per warp
// instruction and kept the L1 pipe saturated.  16-byte chunk q of row r sits
// at chunk q ^ (r mod 16), so the copy and each thread's row reads are free of
// bank conflicts.  Otherwise each thread loads its own row with the following
// slices in flight.  The outputs are built in shared memory and written out
// whole.
constexpr int kTokItem = 128;
constexpr int kStageChunks = 16;  // 16-byte chunks of a staged row: 128 16-bit values

template <int NC, int DT, int B, int CB, int which, bool Z>
__global__ void __launch_bounds__(kAppendThreads, 5) quant_token32_kernel(AppendArgs a) {
  constexpr int D = 128 * NC, SPR = D / 32, HDR = Z ? 4 : 2;
  constexpr int BB = HDR + 4 * B, ROW = SPR * BB;
  constexpr int CBB = CB ? HDR + 4 * CB : 0, CROW = SPR * CBB;
  constexpr int OUTB = kTokItem * (ROW > CROW ? ROW : CROW);
  // staged rows: one pass, and the stage fits the 48 KB of static shared memory
  constexpr bool STAGED = NC == 1 && OUTB + kTokItem * (16 * kStageChunks + 16) + 64 <= 48 * 1024;
  static_assert(kTokItem == kAppendThreads, "one token row per thread");
  __shared__ __align__(16) uint8_t out[OUTB];
  __shared__ __align__(16) uint4 stage[STAGED ? kTokItem * kStageChunks : 1];
  __shared__ const uint4* rowp[STAGED ? kTokItem : 1];
  __shared__ uint8_t* rowd[kTokItem];  // tiered or paged: each row's destination
  __shared__ uint32_t page_bad;
  const Layout& lo = a.lo;
  const int li = blockIdx.z / lo.B, seq = blockIdx.z % lo.B, h = blockIdx.y;
  const int layer = a.layer0 + li;
  SeqSpan s = read_span(a, seq);
  if (!s.ok) return;
  const int q0 = q_end_of(lo, s.T0), q1 = q_end_of(lo, s.T1), c1 = c_end_of(lo, s.T1);
  const int base = (q0 / kTokItem) * kTokItem + blockIdx.x * kTokItem;
  const int u0 = max(base, q0), u1 = min(base + kTokItem, q1);
  if (u0 >= u1) return;
  const int n_tok = u1 - u0;
  if (threadIdx.x == 0) page_bad = 0;
  const int j = threadIdx.x;
  const int t = u0 + j;
  // tiered chunks start at multiples of 32 (Gamma = 32), and cold rows come
  // before hot rows, so rows of both strides never overlap in the tile
  const bool to_cold = CB != 0 && lo.tiered && t < c1;
  uint8_t* dst = out + j * (to_cold ? CROW : ROW);
  // one 32-value slice: r holds its 16-bit values
  auto slice = [&](const uint4 (&r)[4], int sl) {
    if constexpr (CB == 2 && !Z) {
      if (to_cold) {
        const uint32_t w[16] = {r[0].x, r[0].y, r[0].z, r[0].w, r[1].x, r[1].y, r[1].z, r[1].w,
                                r[2].x, r[2].y, r[2].z, r[2].w, r[3].x, r[3].y, r[3].z, r[3].w};
        if (cold2_slice<DT, B>(w, dst + sl * CBB)) return;
      }
    }
    float v[32], mn = 0.f, mx = 0.f;
    if constexpr (Z) {  // block extremes on the 16-bit pairs
      uint32_t lo2 = r[0].x, hi2 = lo2;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t ww[4] = {r[q].x, r[q].y, r[q].z, r[q].w};
#pragma unroll
        for (int e = (q == 0 ? 1 : 0); e < 4; ++e) {
          lo2 = min2_16<DT>(lo2, ww[e]);
          hi2 = max2_16<DT>(hi2, ww[e]);
        }
      }
      const float2 l = raw_pair_to_f32<DT>(lo2), h = raw_pair_to_f32<DT>(hi2);
      mn = fminf(l.x, l.y);
      mx = fmaxf(h.x, h.y);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t ww[4] = {r[q].x, r[q].y, r[q].z, r[q].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = raw_pair_to_f32<DT>(ww[e]);
        v[8 * q + 2 * e] = f.x;
        v[8 * q + 2 * e + 1] = f.y;
      }
    }
    hot_or_cold<B, CB, Z>(v, to_cold, dst + sl * BB, dst + sl * CBB, mn, mx);
  };
  if constexpr (STAGED) {
    if (j < n_tok)
      rowp[j] = reinterpret_cast<const uint4*>(t < s.T0 ? resid_row(lo, a.cp, which, layer, seq, h, t)
                                                        : input_row(a, which, li, s, h, t));
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kTokItem * kStageChunks / kAppendThreads; ++i) {
      const int f = i * kAppendThreads + threadIdx.x, r = f / kStageChunks, q = f % kStageChunks;
      if (r < n_tok) cp_async16(&stage[r * kStageChunks + (q ^ (r % kStageChunks))], rowp[r] + q);
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    if (j < n_tok) {
#pragma unroll
      for (int sl = 0; sl < SPR; ++sl) {
        uint4 r[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) r[q] = stage[j * kStageChunks + ((4 * sl + q) ^ (j % kStageChunks))];
        slice(r, sl);
      }
    }
  } else if (j < n_tok) {
    const uint4* src = reinterpret_cast<const uint4*>(t < s.T0 ? resid_row(lo, a.cp, which, layer, seq, h, t)
                                                                 : input_row(a, which, li, s, h, t));
    // PF slices of the row in flight: the whole 128-value row, or two slices
    // of a 256-value row
    constexpr int PF = SPR <= 4 ? SPR : 2;
    uint4 r[PF][4];
#pragma unroll
    for (int p = 0; p < PF; ++p)
#pragma unroll
      for (int q = 0; q < 4; ++q) r[p][q] = src[4 * p + q];
#pragma unroll
    for (int sl = 0; sl < SPR; ++sl) {
      uint4 c[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) c[q] = r[sl % PF][q];
      if (sl + PF < SPR) {
#pragma unroll
        for (int q = 0; q < 4; ++q) r[sl % PF][q] = src[4 * (sl + PF) + q];
      }
      slice(c, sl);
    }
  }
  __syncthreads();
  if (!lo.paged && !lo.tiered) {
    bool bad = false;
    uint8_t* dst = main_row(lo, a.cp, which, layer, seq, h, u0, &bad);
    if (span_ok(lo, a.cp, which, dst, (int64_t)n_tok * ROW)) block_copy_out(dst, out, n_tok * ROW);
    return;
  }
  // tiered or paged: thread j finds token row j's destination (a row of a
  // page, of the hot ring or of the cold tier); then the block writes the
  // tile word by word, consecutive threads on consecutive words, so that a
  // run of consecutive rows goes out as whole lines
  if (j < n_tok) {
    bool bad = false;
    uint8_t* d = to_cold ? cold_row(lo, a.cp, which, layer, seq, h, t)
                         : main_row(lo, a.cp, which, layer, seq, h, t, &bad);
    if (bad) page_bad = 1;
    rowd[j] = bad ? nullptr : d;
  }
  __syncthreads();
  const int n_c = CB != 0 && lo.tiered ? min(max(c1 - u0, 0), n_tok) : 0;
  if constexpr (CB != 0) rows_out<CROW / 4>(rowd, out, 0, n_c);
  rows_out<ROW / 4>(rowd, out, n_c, n_tok);
  if (threadIdx.x == 0 && page_bad) atomicOr(a.status, KVQ_DEV_PAGE);
}

// Per-channel blocks over 32-token groups: thread = (group lane, channel
// pair); a block takes NG = GPC x kGroupSteps consecutive groups, each thread
// kGroupSteps of them in turn.  A warp's loads of one token row are 32
// consecutive words (one line), so the rows are read in place.  Each group
// row (D blocks) is built in shared memory and written out whole.
constexpr int kGroupSteps = 2;

// One tier, or symmetric tiers (the pair quantizers and the direct cold rule,
// no 32-value float arrays in line): 72 registers and seven CTAs per SM hide
// more of the load latency; measured faster than five or six CTAs even where
// the asymmetric body spills a few words.
template <int CB, bool Z>
constexpr int channel_ctas() { return CB == 0 || (CB == 2 && !Z) ? 7 : 5; }

template <int NC, int DT, int B, int CB, int which, bool Z>
__global__ void __launch_bounds__(kAppendThreads, channel_ctas<CB, Z>()) quant_channel32_kernel(AppendArgs a) {
  constexpr int D = 128 * NC, PAIRS = D / 2, GPC = kAppendThreads / PAIRS, NG = GPC * kGroupSteps;
  constexpr int HDR = Z ? 4 : 2;
  constexpr int BB = HDR + 4 * B, GROW = D * BB;
  constexpr int CBB = CB ? HDR + 4 * CB : 0, CGROW = D * CBB;
  constexpr int SLOT = GROW > CGROW ? GROW : CGROW;
  __shared__ __align__(16) uint8_t out[NG * SLOT];
  const Layout& lo = a.lo;
  const int li = blockIdx.z / lo.B, seq = blockIdx.z % lo.B, h = blockIdx.y;
  const int layer = a.layer0 + li;
  SeqSpan s = read_span(a, seq);
  if (!s.ok) return;
  const int q0 = q_end_of(lo, s.T0), q1 = q_end_of(lo, s.T1), c1 = c_end_of(lo, s.T1);
  const int base = (q0 / (kTile * NG)) * (kTile * NG) + blockIdx.x * (kTile * NG);
  if (base + kTile * NG <= q0 || base >= q1) return;
  const int gl = threadIdx.x / PAIRS, cp = threadIdx.x % PAIRS;
  // the rows of group step gs for this thread's channel pair: window ring
  // slots for tokens below T0, new input rows (a fixed stride apart) from T0
  // on; false when the group is outside this call's range
  auto load_group = [&](int gs, uint32_t (&raw)[32]) -> bool {
    const int t0 = base + kTile * (gs * GPC + gl);
    if (t0 < q0 || t0 >= q1) return false;
    const int n_rw = min(max(s.T0 - t0, 0), kTile);  // leading tokens from the window
    const uint32_t* in = nullptr;
    if (n_rw < kTile) in = reinterpret_cast<const uint32_t*>(input_row(a, which, li, s, h, t0 + n_rw)) + cp;
    const int in_stride = lo.H * D / 2;
    if (n_rw == 0) {
#pragma unroll
      for (int j = 0; j < 32; ++j) raw[j] = in[j * in_stride];
    } else {
      const uint32_t* rw = reinterpret_cast<const uint32_t*>(resid_row(lo, a.cp, which, layer, seq, h, 0)) + cp;
      int slot = t0 % lo.ring;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        raw[j] = j < n_rw ? rw[slot * (D / 2)] : in[(j - n_rw) * in_stride];
        slot = slot + 1 == lo.ring ? 0 : slot + 1;
      }
    }
    return true;
  };
  auto quant_group = [&](int gs, const uint32_t (&raw)[32]) {
    const int gi = gs * GPC + gl;
    const int t0 = base + kTile * gi;
    const bool to_cold = CB != 0 && lo.tiered && t0 < c1;
    float2 mn2 = make_float2(0.f, 0.f), mx2 = mn2;
    if constexpr (Z) {  // extremes of both channels' blocks on the 16-bit pairs
      uint32_t lo2 = raw[0], hi2 = raw[0];
#pragma unroll
      for (int j = 1; j < 32; ++j) {
        lo2 = min2_16<DT>(lo2, raw[j]);
        hi2 = max2_16<DT>(hi2, raw[j]);
      }
      mn2 = raw_pair_to_f32<DT>(lo2);
      mx2 = raw_pair_to_f32<DT>(hi2);
      if (!to_cold) {
        block32_zp_x2<DT, B>(raw, mn2, mx2, out + gi * SLOT + 2 * cp * BB, out + gi * SLOT + (2 * cp + 1) * BB);
        return;
      }
    } else if (!to_cold) {
      uint8_t* d0 = out + gi * SLOT + 2 * cp * BB;
      if (!block32_x2<DT, B>(raw, d0, d0 + BB)) {
        uint32_t t[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) t[j] = raw[j];
        block32_pair_slow<DT, B>(t, d0, d0 + BB);
      }
      return;
    }
    if constexpr (CB == 2 && !Z) {  // to_cold
      uint8_t* d0 = out + gi * SLOT + 2 * cp * CBB;
      if (!cold2_x2<DT, B>(raw, d0, d0 + CBB)) {
        uint32_t t[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) t[j] = raw[j];
        cold_pair_slow<DT, B, CB>(t, d0, d0 + CBB);
      }
    } else {
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const uint32_t h16 = hc ? (raw[j] >> 16) : (raw[j] & 0xFFFFu);
          v[j] = in_to_f32_t<DT>(h16);
        }
        const int c = 2 * cp + hc;
        hot_or_cold<B, CB, Z>(v, to_cold, out + gi * SLOT + c * BB, out + gi * SLOT + c * CBB, hc ? mn2.y : mn2.x,
                              hc ? mx2.y : mx2.x);
      }
    }
  };
#pragma unroll 1
  for (int gs = 0; gs < kGroupSteps; ++gs) {
    uint32_t raw[32];
    if (load_group(gs, raw)) quant_group(gs, raw);
  }
  __syncthreads();
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    const int tg = base + kTile * g;
    if (tg < q0 || tg >= q1) continue;
    const bool cold = CB != 0 && lo.tiered && tg < c1;
    bool bad = false;
    uint8_t* dst = cold ? cold_row(lo, a.cp, which, layer, seq, h, tg) : main_row(lo, a.cp, which, layer, seq, h, tg, &bad);
    block_copy_out(dst, out + g * SLOT, cold ? CGROW : GROW);
  }
}

template <int NC, int DT, int B, int CB, bool Z = false>
void launch_token32(const AppendArgs& a, int which, cudaStream_t st) {
  const int chunks = (a.max_new + kTokItem - 1) / kTokItem + 2;
  const dim3 grid(chunks, a.lo.H, a.n_layers * a.lo.B);
  if (which == 0) quant_token32_kernel<NC, DT, B, CB, 0, Z><<<grid, kAppendThreads, 0, st>>>(a);
  else quant_token32_kernel<NC, DT, B, CB, 1, Z><<<grid, kAppendThreads, 0, st>>>(a);
}

template <int NC, int DT, int B, int CB, bool Z = false>
void launch_channel32(const AppendArgs& a, cudaStream_t st) {
  constexpr int span = kTile * (kAppendThreads / (64 * NC)) * kGroupSteps;
  const int chunks = (a.max_new + span - 1) / span + 2;
  quant_channel32_kernel<NC, DT, B, CB, 0, Z><<<dim3(chunks, a.lo.H, a.n_layers * a.lo.B), kAppendThreads, 0, st>>>(a);
}

// Asymmetric formats: launches (or with `dry`, only checks) the specialized
// phase B of tensor `which`; false when none exists.
template <int NC, int DT>
bool launch_fast_zp_tensor(const AppendArgs& a, int which, bool dry, cudaStream_t st) {
  const Layout& lo = a.lo;
  const FmtInfo& f = fmt_main(lo, which);
  const int cb = lo.tiered ? fmt_cold(lo, which).bits : 0;
  if (f.axis == KVQ_AXIS_CHANNEL) {
    if (which != 0) return false;
    if (f.bits == 4 && cb == 0) return dry || (launch_channel32<NC, DT, 4, 0, true>(a, st), true);
    if (f.bits == 4 && cb == 2) return dry || (launch_channel32<NC, DT, 4, 2, true>(a, st), true);
    if (f.bits == 2 && cb == 0) return dry || (launch_channel32<NC, DT, 2, 0, true>(a, st), true);
    return false;
  }
  if (f.bits == 4 && cb == 0) return dry || (launch_token32<NC, DT, 4, 0, true>(a, which, st), true);
  if (f.bits == 2 && cb == 0) return dry || (launch_token32<NC, DT, 2, 0, true>(a, which, st), true);
  if (f.bits == 4 && cb == 2 && which == 1) return dry || (launch_token32<NC, DT, 4, 2, true>(a, which, st), true);
  return false;
}

}  // namespace

// Rotated per-token 128-value formats (4 or 3 bits): launches (or with `dry`,
// only checks) the specialized phase B of tensor `which`.
bool launch_fast_rot(const AppendArgs& a, int which, bool dry, cudaStream_t st);

// Asymmetric-format launchers, one translation unit per input dtype.
bool launch_fast_zp_f16(const AppendArgs& a, int which, bool dry, cudaStream_t st);
bool launch_fast_zp_bf16(const AppendArgs& a, int which, bool dry, cudaStream_t st);

}  // namespace kvq
