// Block quantization, packing and unpacking on the device, plus the warp
// Walsh-Hadamard transform.  The quantizer keeps the fp32 op order of the
// format: amax = max|x|; scale = fp16_rn(min(amax / qmax, 65504));
// code = clamp(rint(x / float(scale)), -qmax, qmax), all codes 0 for a zero
// scale.  Files that quantize are compiled without FMA contraction.
#pragma once

#include "kvq_internal.cuh"

namespace kvq {

// Packed pairs of fp32 (low half = first element).
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t r, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// fp32 bits of 1/sqrt(128): the scale of the orthonormal 128-point transform.
constexpr uint32_t kHadamardScaleBits = 0x3DB504F3u;

__device__ __forceinline__ float hadamard_scale() { return __uint_as_float(kHadamardScaleBits); }

// Unnormalized 128-point fast Walsh-Hadamard transform across one warp:
// lane l holds elements 4l..4l+3.  Radix-2 stages with strides 1, 2, 4, ...,
// 64 in that order; each maps (a, b) = (x[i], x[i+h]) to (a + b, a - b).
__device__ __forceinline__ void warp_fwht128(float v[4]) {
  float a0 = v[0] + v[1], a1 = v[0] - v[1];
  float a2 = v[2] + v[3], a3 = v[2] - v[3];
  v[0] = a0 + a2;
  v[2] = a0 - a2;
  v[1] = a1 + a3;
  v[3] = a1 - a3;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float o = __shfl_xor_sync(0xffffffffu, v[e], m);
      v[e] = upper ? (o - v[e]) : (v[e] + o);
    }
  }
}

// Forward randomized rotation of a 128-chunk held as in warp_fwht128:
// y = d2 * (FWHT(d1 * x) * (1/sqrt(128))).
__device__ __forceinline__ void warp_rotate128(float v[4], const uint32_t* d1, const uint32_t* d2) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int e = 0; e < 4; ++e)
    if ((d1[(4 * lane + e) >> 5] >> ((4 * lane + e) & 31)) & 1u) v[e] = -v[e];
  warp_fwht128(v);
  const float c = hadamard_scale();
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    v[e] = v[e] * c;
    if ((d2[(4 * lane + e) >> 5] >> ((4 * lane + e) & 31)) & 1u) v[e] = -v[e];
  }
}

// Inverse rotation: x = d1 * (FWHT(d2 * y) * (1/sqrt(128))).
__device__ __forceinline__ void warp_unrotate128(float v[4], const uint32_t* d1, const uint32_t* d2) {
  warp_rotate128(v, d2, d1);
}

__device__ __forceinline__ int quant_code(float x, float sf, int qmax) {
  if (sf == 0.0f) return 0;
  float r = rintf(__fdiv_rn(x, sf));
  r = fminf(fmaxf(r, (float)-qmax), (float)qmax);
  return (int)r;
}

// The code of x with one multiply, given rcp = fp32(1/sf) (0 for a zero
// scale).  |x*rcp - fp32(x/sf)| <= 1.5 * 2^-23 * |x/sf| <= 3.5e-5 for the
// quotients a block produces (|x/sf| <= 1.5 qmax, fp16 subnormal scales
// included), so unless the product lies within 2^-14 of a half-integer it
// rounds to the same integer as rint(x / sf); `near` is set otherwise and the
// caller redoes the block with quant_code (the exact IEEE quotient).
__device__ __forceinline__ int code_mul(float x, float rcp, int qmax, bool& near) {
  const float q = x * rcp;
  const float r = rintf(q);
  near |= fabsf(q - r) > 0.49993896484375f;
  return (int)fminf(fmaxf(r, (float)-qmax), (float)qmax);
}

// fp16 scale of a block with absolute maximum amax: fp16_rn(min(amax/qmax, 65504)).
__device__ __forceinline__ __half block_scale_of(float amax, int qmax) {
  return __float2half_rn(fminf(__fdiv_rn(amax, (float)qmax), 65504.0f));
}

// Quantizes G values get(0..G-1) into one block at dst (scale then codes).
// If deq is given, it receives code * scale (exact in fp32).
template <class Get>
__device__ void quant_block_serial(Get get, int G, int bits, uint8_t* dst, float* deq) {
  const int qmax = qmax_of(bits);
  float amax = 0.0f;
  for (int i = 0; i < G; ++i) amax = fmaxf(amax, fabsf(get(i)));
  float s32 = __fdiv_rn(amax, (float)qmax);
  __half s16 = __float2half_rn(fminf(s32, 65504.0f));
  const float sf = __half2float(s16);
  // One 16-bit store (blocks start at even offsets).  Splitting the half's
  // bits into two byte stores was observed to store a value conversion of
  // the scale instead of its low byte with nvcc 13.0 for sm_103a.
  *reinterpret_cast<__half*>(dst) = s16;
  uint8_t* p = dst + 2;
  if (bits == 8) {
    for (int i = 0; i < G; ++i) {
      int c = quant_code(get(i), sf, qmax);
      p[i] = (uint8_t)(c & 0xFF);
      if (deq) deq[i] = (float)c * sf;
    }
  } else if (bits == 4) {
    for (int i = 0; i < G; i += 2) {
      int c0 = quant_code(get(i), sf, qmax), c1 = quant_code(get(i + 1), sf, qmax);
      p[i >> 1] = (uint8_t)((c0 + 8) | ((c1 + 8) << 4));
      if (deq) {
        deq[i] = (float)c0 * sf;
        deq[i + 1] = (float)c1 * sf;
      }
    }
  } else if (bits == 3) {
    for (int i = 0; i < G; i += 8) {
      uint32_t w = 0;
      for (int j = 0; j < 8; ++j) {
        int c = quant_code(get(i + j), sf, qmax);
        w |= (uint32_t)(c + 4) << (3 * j);
        if (deq) deq[i + j] = (float)c * sf;
      }
      uint8_t* q = p + (i >> 3) * 3;
      q[0] = (uint8_t)(w & 0xFF);
      q[1] = (uint8_t)((w >> 8) & 0xFF);
      q[2] = (uint8_t)((w >> 16) & 0xFF);
    }
  } else {  // 2 bits
    for (int i = 0; i < G; i += 4) {
      uint32_t b = 0;
      for (int j = 0; j < 4; ++j) {
        int c = quant_code(get(i + j), sf, qmax);
        b |= (uint32_t)(c + 2) << (2 * j);
        if (deq) deq[i + j] = (float)c * sf;
      }
      p[i >> 2] = (uint8_t)b;
    }
  }
}

// Code i of a block payload (signed).
__device__ __forceinline__ int unpack_code(const uint8_t* p, int bits, int i) {
  if (bits == 8) return (int)(int8_t)p[i];
  if (bits == 4) return (int)((p[i >> 1] >> ((i & 1) * 4)) & 0xF) - 8;
  if (bits == 3) {
    const uint8_t* q = p + (i >> 3) * 3;
    uint32_t w = (uint32_t)q[0] | ((uint32_t)q[1] << 8) | ((uint32_t)q[2] << 16);
    return (int)((w >> (3 * (i & 7))) & 7u) - 4;
  }
  return (int)((p[i >> 2] >> (2 * (i & 3))) & 3u) - 2;
}

// fp16 scale at the start of a block (blocks start at even offsets).
__device__ __forceinline__ float block_scale(const uint8_t* blk) {
  return __half2float(*reinterpret_cast<const __half*>(blk));
}

// Dequantizes a whole block into out[0..G-1] (code * scale, exact).
__device__ __forceinline__ void dequant_block_serial(const uint8_t* blk, int G, int bits, float* out, int stride) {
  const float sf = block_scale(blk);
  for (int i = 0; i < G; ++i) out[i * stride] = (float)unpack_code(blk + 2, bits, i) * sf;
}

// TBQ4 block (fp16 norm, 4-bit centroid indices): element i = cb[index] * norm
// (exact: both factors are fp16 values).
__device__ __forceinline__ void dequant_tbq4_serial(const uint8_t* blk, const float* cb, float* out, int stride) {
  const float n = block_scale(blk);
  for (int i = 0; i < 128; ++i) out[i * stride] = cb[(blk[2 + (i >> 1)] >> ((i & 1) * 4)) & 0xF] * n;
}

// Asymmetric block (fp16 scale, fp16 zero, unbiased codes): element i =
// code * scale + zero in fp32 (the product is exact, the sum rounds once).
__device__ __forceinline__ float zp_value(const uint8_t* blk, int bits, int i) {
  const int c = unpack_code(blk + 4, bits, i) + (bits == 8 ? 0 : 1 << (bits - 1));  // the raw field
  return __fadd_rn(__fmul_rn((float)c, block_scale(blk)), __half2float(*reinterpret_cast<const __half*>(blk + 2)));
}

__device__ __forceinline__ void dequant_zp_serial(const uint8_t* blk, int G, int bits, float* out, int stride) {
  for (int i = 0; i < G; ++i) out[i * stride] = zp_value(blk, bits, i);
}

// Element i of a block (TBQ4, asymmetric or uniform codes), in the stored domain.
__device__ __forceinline__ float block_value(const uint8_t* blk, int bits, int codebook, int zp, const float* cb,
                                             int i) {
  if (codebook) return cb[(blk[2 + (i >> 1)] >> ((i & 1) * 4)) & 0xF] * block_scale(blk);
  if (zp) return zp_value(blk, bits, i);
  return (float)unpack_code(blk + 2, bits, i) * block_scale(blk);
}

// Asymmetric block of 32 values (op order of the format): mn, mx = min, max
// (a zero minimum as +0); s16 = fp16(min((mx - mn) / (2^b - 1), 65504));
// z16 = fp16(mn clipped to +-65504); code = clamp(rint((x - z) / s), 0, 2^b - 1), 0 when s = 0.  The
// block (scale, zero, codes in little-endian b-bit fields) goes to blk when
// given; dq (optional) receives code * s + z.  Not inlined: the generic
// kernels call it from many places and it holds 32 IEEE divides.
static __device__ __noinline__ void quant_zp32_mem(const float* v, int bits, uint8_t* blk, float* dq) {
  const int qlev = (1 << bits) - 1;
  float mn = v[0], mx = v[0];
  for (int j = 1; j < 32; ++j) {
    mn = fminf(mn, v[j]);
    mx = fmaxf(mx, v[j]);
  }
  mn = __fadd_rn(mn, 0.0f);  // a zero minimum is stored as +0
  const __half s16 = __float2half_rn(fminf(__fdiv_rn(__fsub_rn(mx, mn), (float)qlev), 65504.0f));
  const __half z16 = __float2half_rn(fminf(fmaxf(mn, -65504.0f), 65504.0f));
  const float sf = __half2float(s16), zf = __half2float(z16);
  uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int j = 0; j < 32; ++j) {
    int c = 0;
    if (sf != 0.f) c = (int)fminf(fmaxf(rintf(__fdiv_rn(__fsub_rn(v[j], zf), sf)), 0.f), (float)qlev);
    if (dq) dq[j] = __fadd_rn(__fmul_rn((float)c, sf), zf);
    const int bit = bits * j, k = bit / 32, sh = bit % 32;
    w[k] |= (uint32_t)c << sh;
    if (sh + bits > 32) w[k + 1] |= (uint32_t)c >> (32 - sh);
  }
  if (!blk) return;
  uint16_t* p = reinterpret_cast<uint16_t*>(blk);
  p[0] = __half_as_ushort(s16);
  p[1] = __half_as_ushort(z16);
  for (int k = 0; k < bits; ++k) {
    p[2 + 2 * k] = (uint16_t)w[k];
    p[3 + 2 * k] = (uint16_t)(w[k] >> 16);
  }
}

// Array form of quant_zp32_mem: passes a copy, so that the caller's array
// keeps its registers.
__device__ __forceinline__ void quant_zp32(const float (&v)[32], int bits, uint8_t* blk, float* dq) {
  float t[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) t[j] = v[j];
  quant_zp32_mem(t, bits, blk, dq);
}

// Index of u among the 15 ascending thresholds: how many lie strictly below.
__device__ __forceinline__ uint32_t tbq4_index(float u, const float* t) {
  uint32_t k = 0;
#pragma unroll
  for (int j = 0; j < 15; ++j) k += u > t[j] ? 1u : 0u;
  return k;
}

}  // namespace kvq
