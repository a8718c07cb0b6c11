// The three phases of quantize-on-append for every format, as device
// functions over one unit: tile `bx` of (layer index li, sequence seq, kv
// head h), with the calling block's kAppendThreads threads.  The append
// kernels wrap them one block per unit; the fused decode step calls them for
// the tiles a single new token changes.  Every rounding step is an explicit
// intrinsic or a lone multiply or add, so the codes do not depend on the
// including file's FMA-contraction setting.
//
//   A  hot groups [c_end(T0), min(c_end(T1), q_end(T0))) requantized to the
//      cold format from their dequantized hot values;
//   B  units [q_end(T0), q_end(T1)) quantized from the window (tokens < T0)
//      or the new input; units below c_end(T1) continue to the cold format
//      through the same hot quantize -> dequantize -> requantize;
//   C  new tokens in [max(T0, q_end(T1)), T1) copied into the window ring.
#pragma once

#include "append_common.cuh"

namespace kvq {
namespace {

// ---- per-token rows: one warp per (token, kv head) ----------------------------
//
// Lane l holds channels 128c + 4l .. 128c + 4l + 3 of every 128-chunk c (the
// layout of warp_rotate128), NC = D / 128 chunks.

template <int NC>
__device__ __forceinline__ void load_row(const uint16_t* src, int dtype, float (&v)[NC][4]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const uint2 w = *reinterpret_cast<const uint2*>(src + 128 * c + 4 * lane);
    v[c][0] = in_to_f32((uint16_t)(w.x & 0xFFFF), dtype);
    v[c][1] = in_to_f32((uint16_t)(w.x >> 16), dtype);
    v[c][2] = in_to_f32((uint16_t)(w.y & 0xFFFF), dtype);
    v[c][3] = in_to_f32((uint16_t)(w.y >> 16), dtype);
  }
}

// Quantizes the warp's row into `row` (skipped when row is null) with blocks
// of G channels and `bits` bits; dq (optional) receives code * scale.
template <int NC>
__device__ __forceinline__ void warp_quant_row(const float (&v)[NC][4], int G, int bits, uint8_t* row,
                                               float (*dq)[4]) {
  const int lane = threadIdx.x & 31;
  const int qmax = qmax_of(bits);
  const int bb = block_bytes_of(bits, G);
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    float m = fmaxf(fmaxf(fabsf(v[c][0]), fabsf(v[c][1])), fmaxf(fabsf(v[c][2]), fabsf(v[c][3])));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
    if (G == 128) {
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
    }
    const __half s16 = block_scale_of(m, qmax);
    const float sf = __half2float(s16);
    const float rcp = sf == 0.f ? 0.f : __frcp_rn(sf);
    int code[4];
    bool near = false;
#pragma unroll
    for (int e = 0; e < 4; ++e) code[e] = code_mul(v[c][e], rcp, qmax, near);
    if (__any_sync(0xffffffffu, near)) {
#pragma unroll
      for (int e = 0; e < 4; ++e) code[e] = quant_code(v[c][e], sf, qmax);
    }
    if (dq) {
#pragma unroll
      for (int e = 0; e < 4; ++e) dq[c][e] = (float)code[e] * sf;
    }
    const int ch0 = 128 * c + 4 * lane;
    const int pos = ch0 % G;
    uint8_t* blk = row ? row + (ch0 / G) * bb : nullptr;
    if (bits == 3) {  // 12 bits per lane; even lanes write the 24-bit word of a lane pair
      uint32_t w12 = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) w12 |= (uint32_t)(code[e] + 4) << (3 * e);
      const uint32_t other = __shfl_xor_sync(0xffffffffu, w12, 1);
      if (blk && !(lane & 1)) {
        const uint32_t w = w12 | (other << 12);
        uint8_t* p = blk + 2 + (pos / 8) * 3;
        p[0] = (uint8_t)(w & 0xFFu);
        p[1] = (uint8_t)((w >> 8) & 0xFFu);
        p[2] = (uint8_t)((w >> 16) & 0xFFu);
      }
    }
    if (!blk) continue;
    if (pos == 0) *reinterpret_cast<__half*>(blk) = s16;
    uint8_t* p = blk + 2;
    if (bits == 8) {
      *reinterpret_cast<uint16_t*>(p + pos) = (uint16_t)((code[0] & 0xFF) | ((code[1] & 0xFF) << 8));
      *reinterpret_cast<uint16_t*>(p + pos + 2) = (uint16_t)((code[2] & 0xFF) | ((code[3] & 0xFF) << 8));
    } else if (bits == 4) {
      *reinterpret_cast<uint16_t*>(p + pos / 2) =
          (uint16_t)((code[0] + 8) | ((code[1] + 8) << 4) | ((code[2] + 8) << 8) | ((code[3] + 8) << 12));
    } else if (bits == 2) {
      p[pos / 4] = (uint8_t)((code[0] + 2) | ((code[1] + 2) << 2) | ((code[2] + 2) << 4) | ((code[3] + 2) << 6));
    }
  }
}

// ---- per-channel groups: one thread per channel, 32 tokens -----------------

// The 32 codes of one per-channel block as a little-endian bit stream of
// 32*B bits (code j, with its storage bias, at bit B*j; int8 two's
// complement for B = 8): the byte layout of every packing of the format.
template <int B, bool EXACT>
__device__ __forceinline__ bool channel_stream(const float (&v)[32], float sf, float rcp, uint32_t (&w)[B],
                                               float* dq) {
  constexpr int qmax = (1 << (B - 1)) - 1;
  bool near = false;
#pragma unroll
  for (int k = 0; k < B; ++k) w[k] = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int c = EXACT ? quant_code(v[j], sf, qmax) : code_mul(v[j], rcp, qmax, near);
    if (dq) dq[j] = (float)c * sf;
    const uint32_t u = B == 8 ? (uint32_t)(c & 0xFF) : (uint32_t)(c + qmax + 1);
    const int bit = B * j, k = bit / 32, sh = bit % 32;
    w[k] |= u << sh;
    if (sh + B > 32) w[k + 1] |= u >> (32 - sh);
  }
  return near;
}

template <int B>
__device__ __forceinline__ void channel_block(const float (&v)[32], float m, uint8_t* blk, float* dq) {
  const __half s16 = block_scale_of(m, (1 << (B - 1)) - 1);
  const float sf = __half2float(s16);
  const float rcp = sf == 0.f ? 0.f : __frcp_rn(sf);
  uint32_t w[B];
  if (channel_stream<B, false>(v, sf, rcp, w, dq)) channel_stream<B, true>(v, sf, rcp, w, dq);
  if (!blk) return;
  *reinterpret_cast<__half*>(blk) = s16;
  uint16_t* p = reinterpret_cast<uint16_t*>(blk + 2);
#pragma unroll
  for (int k = 0; k < B; ++k) {
    p[2 * k] = (uint16_t)w[k];
    p[2 * k + 1] = (uint16_t)(w[k] >> 16);
  }
}

// Quantizes x[0], x[ld], ..., x[31 ld] (one channel over the group's tokens)
// into the block at blk (skipped when null); dq (optional) receives
// code * scale.
__device__ __forceinline__ void thread_quant_channel(const float* x, int ld, int bits, uint8_t* blk, float* dq) {
  float v[32];
  float m = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    v[j] = x[j * ld];
    m = fmaxf(m, fabsf(v[j]));
  }
  switch (bits) {
    case 8: channel_block<8>(v, m, blk, dq); break;
    case 4: channel_block<4>(v, m, blk, dq); break;
    case 3: channel_block<3>(v, m, blk, dq); break;
    default: channel_block<2>(v, m, blk, dq); break;
  }
}

__device__ __forceinline__ float4 f16x4_to_f32(uint2 w, int dtype) {
  return make_float4(in_to_f32((uint16_t)(w.x & 0xFFFF), dtype), in_to_f32((uint16_t)(w.x >> 16), dtype),
                     in_to_f32((uint16_t)(w.y & 0xFFFF), dtype), in_to_f32((uint16_t)(w.y >> 16), dtype));
}

// 32 values v[] of one block slice quantized with the scale of block absolute
// maximum m (shared by the threads of a 128-value block); the payload
// (32*B bits) goes to dst, the scale to blk when blk is given; dq (optional)
// receives code * scale.
template <int B>
__device__ __forceinline__ void quant32(const float (&v)[32], float m, uint8_t* blk, uint8_t* dst, float* dq) {
  const __half s16 = block_scale_of(m, (1 << (B - 1)) - 1);
  const float sf = __half2float(s16);
  const float rcp = sf == 0.f ? 0.f : __frcp_rn(sf);
  uint32_t w[B];
  if (channel_stream<B, false>(v, sf, rcp, w, dq)) channel_stream<B, true>(v, sf, rcp, w, dq);
  if (blk) *reinterpret_cast<__half*>(blk) = s16;
  if (!dst) return;
  uint16_t* p = reinterpret_cast<uint16_t*>(dst);
#pragma unroll
  for (int k = 0; k < B; ++k) {
    p[2 * k] = (uint16_t)w[k];
    p[2 * k + 1] = (uint16_t)(w[k] >> 16);
  }
}

__device__ __forceinline__ void quant32_bits(int bits, const float (&v)[32], float m, uint8_t* blk, uint8_t* dst,
                                             float* dq) {
  switch (bits) {
    case 8: quant32<8>(v, m, blk, dst, dq); break;
    case 4: quant32<4>(v, m, blk, dst, dq); break;
    case 3: quant32<3>(v, m, blk, dst, dq); break;
    default: quant32<2>(v, m, blk, dst, dq); break;
  }
}

__device__ __forceinline__ float amax32(const float (&v)[32]) {
  float m = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) m = fmaxf(m, fabsf(v[j]));
  return m;
}

// Phase B: quantize units [q_end(T0), q_end(T1)).  The chunk's K and V rows
// are copied to shared memory as raw 16-bit values (cp.async); rotated
// formats then pass each row through the randomized Hadamard transform into an
// fp32 tile (one warp per row).  Every thread then quantizes 32 values: one
// channel over the group's tokens (per-channel blocks) or a 32-value slice of
// a token row (per-token blocks; the 4 slices of a 128-value block are
// neighbouring lanes that combine their absolute maxima).
template <int NC, bool ROT>
__device__ __forceinline__ void append_quantize_unit(const AppendArgs& a, int li, int seq, int h, int bx,
                                                     uint8_t* sm) {
  constexpr int D = 128 * NC;
  constexpr int RH = D + 8;    // raw row stride in 16-bit values (16-byte multiple, offset banks)
  constexpr int LDF = D + 1;   // fp32 rotated tile stride
  constexpr int SUB = D / 32;  // 32-value slices per row
  uint16_t* raw = reinterpret_cast<uint16_t*>(sm);                          // [2][kTile][RH]
  float* fl = reinterpret_cast<float*>(sm + 2 * kTile * RH * sizeof(uint16_t));  // [2][kTile][LDF] (ROT)
  __shared__ uint32_t page_bad;
  const Layout& lo = a.lo;
  const int layer = a.layer0 + li;
  SeqSpan s = read_span(a, seq);
  if (!s.ok) return;
  const int q0 = q_end_of(lo, s.T0), q1 = q_end_of(lo, s.T1), c1 = c_end_of(lo, s.T1);
  const int base = (q0 / kTile) * kTile + bx * kTile;
  const int u0 = max(base, q0), u1 = min(base + kTile, q1);
  if (u0 >= u1) return;
  const int n_tok = u1 - u0;
  const bool to_cold = lo.tiered && u0 < c1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  if (tid == 0) page_bad = 0;

  // 1. raw rows -> shared memory
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    for (int e = tid; e < n_tok * (D / 8); e += blockDim.x) {
      const int j = e / (D / 8), c8 = e % (D / 8), t = u0 + j;
      const uint16_t* src = t < s.T0 ? resid_row(lo, a.cp, which, layer, seq, h, t) : input_row(a, which, li, s, h, t);
      cp_async16(raw + (which * kTile + j) * RH + 8 * c8, src + 8 * c8);
    }
  }
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  bool rot[2] = {(lo.flags & KVQ_ROTATE_K) != 0, (lo.flags & KVQ_ROTATE_V) != 0};
  if constexpr (ROT) {
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      if (!rot[which]) continue;
      for (int j = warp; j < n_tok; j += kAppendThreads / 32) {
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const uint2 w = *reinterpret_cast<const uint2*>(raw + (which * kTile + j) * RH + 128 * c + 4 * lane);
          const float4 x = f16x4_to_f32(w, lo.dtype);
          float v[4] = {x.x, x.y, x.z, x.w};
          warp_rotate128(v, lo.d1, lo.d2);
          float* dst = fl + (which * kTile + j) * LDF + 128 * c + 4 * lane;
          dst[0] = v[0];
          dst[1] = v[1];
          dst[2] = v[2];
          dst[3] = v[3];
        }
      }
    }
    __syncthreads();
  }

  // 2. quantize
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const FmtInfo& f = fmt_main(lo, which);
    const FmtInfo& fc = fmt_cold(lo, which);
    const uint16_t* rt = raw + which * kTile * RH;
    if (f.axis == KVQ_AXIS_CHANNEL) {
      // one group of 32 tokens; thread = channel
      for (int c = tid; c < D; c += blockDim.x) {
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = in_to_f32(rt[j * RH + c], lo.dtype);
        if (f.zp) {  // asymmetric blocks
          bool bad = false;
          if (to_cold) {
            float dq[32];
            quant_zp32(v, f.bits, nullptr, dq);
            quant_zp32(dq, fc.bits, cold_row(lo, a.cp, which, layer, seq, h, u0) + (int64_t)c * fc.bb, nullptr);
          } else {
            quant_zp32(v, f.bits, main_row(lo, a.cp, which, layer, seq, h, u0, &bad) + (int64_t)c * f.bb, nullptr);
          }
          continue;
        }
        const float m = amax32(v);
        if (to_cold) {
          float dq[32];
          quant32_bits(f.bits, v, m, nullptr, nullptr, dq);
          uint8_t* blk = cold_row(lo, a.cp, which, layer, seq, h, u0) + (int64_t)c * fc.bb;
          quant32_bits(fc.bits, dq, amax32(dq), blk, blk + 2, nullptr);
        } else {
          bool bad = false;
          uint8_t* blk = main_row(lo, a.cp, which, layer, seq, h, u0, &bad) + (int64_t)c * f.bb;
          quant32_bits(f.bits, v, m, blk, blk + 2, nullptr);
        }
      }
      continue;
    }
    // per-token: thread = (row, 32-value slice).  32-value blocks: lane = row
    // (conflict-free reads); 128-value blocks: the 4 slices of a block are
    // neighbouring lanes.  Every lane runs the loop so that the exchange of
    // 128-value block maxima stays warp-uniform.
    const int spb = f.group / 32;
    for (int u = tid; u < kTile * SUB; u += blockDim.x) {
      const int j = spb == 1 ? (u % kTile) : (u / SUB);
      const int sl = spb == 1 ? (u / kTile) : (u % SUB);
      const bool valid = j < n_tok;
      float v[32];
      if (ROT && rot[which]) {
        const float* x = fl + (which * kTile + j) * LDF + 32 * sl;
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = valid ? x[e] : 0.f;
      } else {
        const uint4* x = reinterpret_cast<const uint4*>(rt + j * RH + 32 * sl);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 w = valid ? x[k] : make_uint4(0, 0, 0, 0);
          const float4 a0 = f16x4_to_f32(make_uint2(w.x, w.y), lo.dtype);
          const float4 a1 = f16x4_to_f32(make_uint2(w.z, w.w), lo.dtype);
          v[8 * k + 0] = a0.x;
          v[8 * k + 1] = a0.y;
          v[8 * k + 2] = a0.z;
          v[8 * k + 3] = a0.w;
          v[8 * k + 4] = a1.x;
          v[8 * k + 5] = a1.y;
          v[8 * k + 6] = a1.z;
          v[8 * k + 7] = a1.w;
        }
      }
      float m = amax32(v);
      if (spb == 4) {
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
      }
      // TBQ4: sum of squares of the 128-value block, in the format's order
      // (each slice in index order, then (s0 + s1) + (s2 + s3))
      float ss = 0.f;
      if (f.codebook) {
#pragma unroll
        for (int e = 0; e < 32; ++e) ss = __fadd_rn(ss, __fmul_rn(v[e], v[e]));
        ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, 1));
        ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, 2));
      }
      if (!valid) continue;
      const int t = u0 + j;
      const int b = sl / spb, within = sl % spb;  // block, slice within the block
      if (f.codebook) {
        bool bad = false;
        uint8_t* row = main_row(lo, a.cp, which, layer, seq, h, t, &bad);
        if (bad) {
          page_bad = 1;
          continue;
        }
        uint8_t* blk = row + b * f.bb;
        const __half n16 = __float2half_rn(fminf(__fsqrt_rn(ss), 65504.0f));
        const float nf = __half2float(n16);
        uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float u = nf > 0.f ? __fdiv_rn(v[e], nf) : 0.f;
          w[e >> 3] |= tbq4_index(u, lo.cbt) << (4 * (e & 7));
        }
        if (within == 0) *reinterpret_cast<__half*>(blk) = n16;
        uint16_t* p = reinterpret_cast<uint16_t*>(blk + 2 + within * 16);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          p[2 * k] = (uint16_t)w[k];
          p[2 * k + 1] = (uint16_t)(w[k] >> 16);
        }
        continue;
      }
      if (f.zp) {  // asymmetric 32-value blocks
        if (to_cold) {
          float dq[32];
          quant_zp32(v, f.bits, nullptr, dq);
          quant_zp32(dq, fc.bits, cold_row(lo, a.cp, which, layer, seq, h, t) + b * fc.bb, nullptr);
        } else {
          bool bad = false;
          uint8_t* row = main_row(lo, a.cp, which, layer, seq, h, t, &bad);
          if (bad) {
            page_bad = 1;
            continue;
          }
          quant_zp32(v, f.bits, row + b * f.bb, nullptr);
        }
        continue;
      }
      if (to_cold) {
        // tiers keep the hot group size; per-token tiers use 32-value blocks
        float dq[32];
        quant32_bits(f.bits, v, m, nullptr, nullptr, dq);
        uint8_t* blk = cold_row(lo, a.cp, which, layer, seq, h, t) + b * fc.bb;
        quant32_bits(fc.bits, dq, amax32(dq), blk, blk + 2, nullptr);
      } else {
        bool bad = false;
        uint8_t* row = main_row(lo, a.cp, which, layer, seq, h, t, &bad);
        if (bad) {
          page_bad = 1;
          continue;
        }
        uint8_t* blk = row + b * f.bb;
        quant32_bits(f.bits, v, m, within == 0 ? blk : nullptr, blk + 2 + within * 4 * f.bits, nullptr);
      }
    }
  }
  __syncthreads();
  if (tid == 0 && page_bad) atomicOr(a.status, KVQ_DEV_PAGE);
}

// Phase A: hot units [c_end(T0), min(c_end(T1), q_end(T0))) -> cold, from the
// exact dequantized hot values.
template <int NC>
__device__ __forceinline__ void append_requant_unit(const AppendArgs& a, int li, int seq, int h, int bx) {
  const Layout& lo = a.lo;
  constexpr int D = 128 * NC;
  const int layer = a.layer0 + li;
  SeqSpan s = read_span(a, seq);
  if (!s.ok) return;
  const int c0 = c_end_of(lo, s.T0), c1 = c_end_of(lo, s.T1), q0 = q_end_of(lo, s.T0);
  const int stop = min(c1, q0);
  const int u0 = c0 + bx * kTile;  // c0 and units are whole groups (Gamma = 32)
  if (u0 >= stop) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  for (int which = 0; which < 2; ++which) {
    const FmtInfo& f = fmt_main(lo, which);
    const FmtInfo& fc = fmt_cold(lo, which);
    bool bad = false;
    if (f.axis == KVQ_AXIS_CHANNEL) {
      const uint8_t* row = main_row(lo, a.cp, which, layer, seq, h, u0, &bad);
      uint8_t* dst = cold_row(lo, a.cp, which, layer, seq, h, u0);
      for (int c = threadIdx.x; c < D; c += blockDim.x) {
        float x[32];
        if (f.zp) {
          dequant_zp_serial(row + (int64_t)c * f.bb, 32, f.bits, x, 1);
          quant_zp32(x, fc.bits, dst + (int64_t)c * fc.bb, nullptr);
          continue;
        }
        dequant_block_serial(row + (int64_t)c * f.bb, f.group, f.bits, x, 1);
        thread_quant_channel(x, 1, fc.bits, dst + (int64_t)c * fc.bb, nullptr);
      }
      continue;
    }
    if (f.zp) {  // per-token asymmetric 32-value blocks: thread = (token, block)
      for (int item = threadIdx.x; item < kTile * (D / 32); item += blockDim.x) {
        const int j = item / (D / 32), b = item % (D / 32);
        const uint8_t* row = main_row(lo, a.cp, which, layer, seq, h, u0 + j, &bad);
        if (!row) continue;
        float x[32];
        dequant_zp_serial(row + b * f.bb, 32, f.bits, x, 1);
        quant_zp32(x, fc.bits, cold_row(lo, a.cp, which, layer, seq, h, u0 + j) + b * fc.bb, nullptr);
      }
      continue;
    }
    for (int j = warp; j < kTile; j += nw) {
      const uint8_t* row = main_row(lo, a.cp, which, layer, seq, h, u0 + j, &bad);
      float v[NC][4];
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const int ch0 = 128 * c + 4 * lane;
        const uint8_t* blk = row + (ch0 / f.group) * f.bb;
        const float sf = block_scale(blk);
#pragma unroll
        for (int e = 0; e < 4; ++e) v[c][e] = (float)unpack_code(blk + 2, f.bits, ch0 % f.group + e) * sf;
      }
      warp_quant_row<NC>(v, fc.group, fc.bits, cold_row(lo, a.cp, which, layer, seq, h, u0 + j), nullptr);
    }
  }
}

// Phase C: new tokens that stay in the 16-bit window.
__device__ __forceinline__ void append_window_unit(const AppendArgs& a, int li, int seq, int h, int bx) {
  const Layout& lo = a.lo;
  const int layer = a.layer0 + li;
  SeqSpan s = read_span(a, seq);
  if (!s.ok) return;
  // at most R + Gamma - 1 tokens stay in the window: the grid covers that
  // span from its first token
  const int w0 = max(s.T0, q_end_of(lo, s.T1));
  const int ta = w0 + bx * kTile, tb = min(ta + kTile, s.T1);
  if (ta >= tb) return;
  const int halfD = lo.D / 2;
  for (int which = 0; which < 2; ++which) {
    for (int e = threadIdx.x; e < (tb - ta) * halfD; e += blockDim.x) {
      const int t = ta + e / halfD, d2 = e % halfD;
      const uint32_t* src = (const uint32_t*)input_row(a, which, li, s, h, t);
      uint32_t* dst = (uint32_t*)resid_row(lo, a.cp, which, layer, seq, h, t);
      dst[d2] = src[d2];
    }
  }
}

}  // namespace
}  // namespace kvq
