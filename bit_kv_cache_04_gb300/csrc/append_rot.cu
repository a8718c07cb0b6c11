// Quantize-on-append for rotated per-token formats (randomized Hadamard
// transform of every 128-value chunk, then one fp16 scale and 4- or 3-bit
// codes per 128 values: the 66 B / 128 and 50 B / 128 blocks of trefon.com,
// "Matematyka cache KV", section "Jak 4-bitowemu cache to uchodzi: najpierw
// obrot").  Compiled with --fmad=false like the other append kernels.
//
// Layout: four lanes take one 128-value chunk, lane a4 = lane % 4 holding the
// 32 consecutive values 32 a4 .. 32 a4 + 31, so a warp holds eight chunks (eight
// tokens at D = 128, four at D = 256).  The transform keeps the format's
// stage order (strides 1, 2, ..., 64; (a, b) -> (a + b, a - b)): strides
// 1..16 run inside a lane, 32 and 64 across the four lanes with one shuffle
// per value each.  Stride 1 runs on scalars; its outputs form pairs
// (x[2i], x[2i+1]) on which the other six stages and the quantizer's
// multiply and adds run as packed fp32x2 operations (each half rounded like
// the scalar operation).  d1 flips the sign bits of the 16-bit inputs.  With t
// the unnormalized transform and c = 1/sqrt(128), the format's value is
// y = d2 RN(t c) and its code rint(RN(y / s)).  Rounding to nearest (and to
// even at ties) is odd-symmetric, so code(y) = d2 code(RN(t c)): the codes are
// taken on t and d2 negates the packed fields at the end.  The four lanes of a
// chunk combine their absolute maxima (max |RN(t c)| = RN(max |t| c), rounding
// being monotonic), and each lane quantizes its 32 values with
// q = RN(t RN(c RN(1/s))): within 5 * 2^-24 |q| of RN(RN(t c) / s), at most
// 2^-18.7 below 8 (|y / s| <= qmax (1 + 2^-10) for normal fp16 scales).  A
// 32-value slice with any q within 2^-16 of a half step, or with a subnormal
// or saturated scale (where x is clamped to +-qmax s first), is redone with
// the exact quotient.  Rows are built in shared memory and written out whole.
//
// TBQ4 blocks (same 66 B: fp16 L2 norm, 4-bit indices into the 16-entry
// Lloyd-Max table; trefon.com, same section): a lane's 32 consecutive values
// are exactly one of the norm's partial sums p_k (index order), S = (p0 + p1)
// + (p2 + p3) by two shuffles, u = RN(y / norm), and the index counts the table
// midpoints strictly below u by one lookup in a binned table
// (tbq4_bins.cuh).  The quotient comes from Markstein's correction step on
// fp32x2 pairs, exact when the norm is 0 (u = 0: rcp = 0 gives +-0) or below
// 65504 (every y finite) and every |y| is at least 2^-100 (the remainder
// y - q0 norm is then exact and the quotient normal); a lane outside those
// bounds divides with the IEEE divide.
#include "append_fast.cuh"
#include "tbq4_bins.cuh"

namespace kvq {
namespace {

constexpr int kRotItem = 128;  // tokens per CTA
constexpr float kNearHalf = 0.5f - 1.52587890625e-05f;  // 1/2 - 2^-16

// Codes of 32 values as a 32*B-bit little-endian stream of biased codes.
// Fast: q = RN(v[j] f[j]) (f[j] the value's factor over the scale).  EXACT:
// y = RN(v[j] g[j]) clamped to +-lim, q = RN(y / sf).  Returns the largest
// distance of a fast q from its rounded integer (0 for EXACT).
template <int B, bool EXACT, class F, class G>
__device__ __forceinline__ float rot_codes(const float (&v)[32], F f, G g, float lim, float sf, uint32_t (&w)[B]) {
  constexpr float magic = kRoundMagic + (float)(1 << (B - 1));
  uint32_t corr[B];
#pragma unroll
  for (int k = 0; k < B; ++k) w[k] = corr[k] = 0;
  float dmax = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    float q;
    if constexpr (EXACT) {
      const float y = fminf(fmaxf(__fmul_rn(v[j], g(j)), -lim), lim);
      q = sf == 0.f ? 0.f : __fdiv_rn(y, sf);
    } else {
      q = __fmul_rn(v[j], f(j));
    }
    const float r = __fadd_rn(q, magic);
    if (!EXACT) dmax = fmaxf(dmax, fabsf(__fsub_rn(q, __fsub_rn(r, magic))));
    const uint32_t bits = __float_as_uint(r);
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
#pragma unroll
  for (int k = 0; k < B; ++k) w[k] -= corr[k];
  return dmax;
}

// Copies `bytes` (even) from shared `src` (16-byte aligned) to global `dst`
// with all threads of the block, in the widest words both ends allow.
__device__ __forceinline__ void copy_out_any(uint8_t* dst, const uint8_t* src, int bytes) {
  const uintptr_t al = reinterpret_cast<uintptr_t>(dst) | (uintptr_t)bytes;
  if ((al & 15u) == 0) {
    for (int e = threadIdx.x; e < bytes / 16; e += blockDim.x)
      reinterpret_cast<uint4*>(dst)[e] = reinterpret_cast<const uint4*>(src)[e];
  } else if ((al & 3u) == 0) {
    for (int e = threadIdx.x; e < bytes / 4; e += blockDim.x)
      reinterpret_cast<uint32_t*>(dst)[e] = reinterpret_cast<const uint32_t*>(src)[e];
  } else {
    for (int e = threadIdx.x; e < bytes / 2; e += blockDim.x)
      reinterpret_cast<uint16_t*>(dst)[e] = reinterpret_cast<const uint16_t*>(src)[e];
  }
}

// Fast codes of the 32 values held as 16 pairs P (t, before the scale):
// q = RN(t crc), r = RN(q + magic); returns the largest |q - rint(q)|.
template <int B>
__device__ __forceinline__ float rot_codes_packed(const uint64_t (&P)[16], float crc, uint32_t (&w)[B]) {
  constexpr float magic = kRoundMagic + (float)(1 << (B - 1));
  const uint64_t C2 = pk2(crc, crc), M2 = pk2(magic, magic);
  uint32_t corr[B];
#pragma unroll
  for (int k = 0; k < B; ++k) w[k] = corr[k] = 0;
  float dmax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint64_t Q = mul2(P[i], C2);
    const uint64_t R = add2(Q, M2);
    float d0, d1, r0, r1;
    upk2(sub2(Q, sub2(R, M2)), d0, d1);
    dmax = fmaxf(dmax, fmaxf(fabsf(d0), fabsf(d1)));
    upk2(R, r0, r1);
    const float rr[2] = {r0, r1};
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const uint32_t bits = __float_as_uint(rr[c]);
      const int bit = B * (2 * i + c), k = bit / 32, sh = bit % 32;
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
  for (int k = 0; k < B; ++k) w[k] -= corr[k];
  return dmax;
}

template <int NC, int DT, int B, int which, bool TQ>
__global__ void __launch_bounds__(kAppendThreads) quant_rot128_kernel(AppendArgs a) {
  constexpr int BB = 2 + 16 * B;  // 66 or 50 bytes per 128 values
  constexpr int ROW = NC * BB;
  constexpr int TPS = 8 / NC;                                // tokens per warp step
  constexpr int WTOK = kRotItem / (kAppendThreads / 32);     // tokens per warp
  constexpr int STEPS = WTOK / TPS;
  constexpr int qmax = (1 << (B - 1)) - 1;
  static_assert(kAppendThreads == 128 && WTOK % TPS == 0, "tile geometry");
  __shared__ __align__(16) uint8_t out[kRotItem * ROW];
  __shared__ uint32_t page_bad;
  __shared__ float2 tbin[2 * kTbqBins];  // TBQ4 lookup: (midpoint inside, count below) per bin
  const Layout& lo = a.lo;
  const int li = blockIdx.z / lo.B, seq = blockIdx.z % lo.B, h = blockIdx.y;
  const int layer = a.layer0 + li;
  SeqSpan s = read_span(a, seq);
  if (!s.ok) return;
  const int q0 = q_end_of(lo, s.T0), q1 = q_end_of(lo, s.T1);
  const int base = (q0 / kRotItem) * kRotItem + blockIdx.x * kRotItem;
  const int u0 = max(base, q0), u1 = min(base + kRotItem, q1);
  if (u0 >= u1) return;
  const int n_tok = u1 - u0;
  if (threadIdx.x == 0) page_bad = 0;
  int k0 = 0;
  if constexpr (TQ) {
    k0 = tbq4_bin_k0(lo.cbt);
    if (threadIdx.x < 2 * kTbqBins) {
      float th;
      int base;
      tbq4_bin_entry(lo.cbt, k0, threadIdx.x, &th, &base);
      tbin[threadIdx.x] = make_float2(th, __int_as_float(base));
    }
    __syncthreads();
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int a4 = lane & 3, slot = lane >> 2;
  const int tok_in_step = slot / NC, chunk = slot % NC;

  // sign constants of this lane's 32 indices 32 a4 + b
  const uint32_t d1w = lo.d1[a4], d2w = lo.d2[a4];
  uint32_t m1[16];  // d1 as sign bits of the 16-bit pairs (b, b + 1)
#pragma unroll
  for (int p = 0; p < 16; ++p) m1[p] = ((d1w >> (2 * p)) & 1u) << 15 | ((d1w >> (2 * p + 1)) & 1u) << 31;
  // d2 in the code domain: a field f of a value with d2 = -1 becomes
  // 2^B - f = (f ^ (2^B - 1)) + 1 (biased codes are >= 1, so no field
  // overflows): negx holds the fields' bits, negl their lowest bits
  uint32_t negx[B], negl[B];
  if constexpr (B == 4) {
    // word k holds values 8k .. 8k + 7: their d2 bits spread to nibble
    // starts (0, 4, ..., 28), then each made a whole nibble
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t x = (d2w >> (8 * k)) & 0xFFu;
      x = (x | (x << 12)) & 0x000F000Fu;
      x = (x | (x << 6)) & 0x03030303u;
      x = (x | (x << 3)) & 0x11111111u;
      negl[k] = x;
      negx[k] = x * 15u;
    }
  } else {
#pragma unroll
    for (int k = 0; k < B; ++k) negx[k] = negl[k] = 0;
#pragma unroll
    for (int b = 0; b < 32; ++b) {
      const uint32_t on = (d2w >> b) & 1u;
      const int bit = B * b, k = bit / 32, sh = bit % 32;
      negx[k] |= (on * ((1u << B) - 1)) << sh;
      if (sh + B > 32) negx[k + 1] |= (on * ((1u << B) - 1)) >> (32 - sh);
      negl[k] |= on << sh;
    }
  }

  auto row_src = [&](int t) -> const uint4* {
    const uint16_t* r = t < s.T0 ? resid_row(lo, a.cp, which, layer, seq, h, t) : input_row(a, which, li, s, h, t);
    return reinterpret_cast<const uint4*>(r + 128 * chunk + 32 * a4);
  };
  auto load = [&](int st, uint4 (&r)[4]) {
    const int j = warp * WTOK + st * TPS + tok_in_step;
    if (j < n_tok) {
      const uint4* src = row_src(u0 + j);
#pragma unroll
      for (int q = 0; q < 4; ++q) r[q] = src[q];
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) r[q] = make_uint4(0, 0, 0, 0);
    }
  };

  uint4 nxt[4];
  load(0, nxt);
#pragma unroll 1
  for (int st = 0; st < STEPS; ++st) {
    if (warp * WTOK + st * TPS >= n_tok) break;  // warp-uniform
    uint4 cur[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) cur[q] = nxt[q];
    if (st + 1 < STEPS) load(st + 1, nxt);
    const int j = warp * WTOK + st * TPS + tok_in_step;

    // d1 on the 16-bit inputs, fp32, stride 1 -> pairs P[i] = (x[2i], x[2i+1])
    uint64_t P[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t ww[4] = {cur[q].x, cur[q].y, cur[q].z, cur[q].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = raw_pair_to_f32<DT>(ww[e] ^ m1[4 * q + e]);
        P[4 * q + e] = pk2(__fadd_rn(f.x, f.y), __fsub_rn(f.x, f.y));
      }
    }
    // strides 2..16 inside the lane (pair strides 1..8)
#pragma unroll
    for (int hp = 1; hp < 16; hp <<= 1) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if (i & hp) continue;
        const uint64_t x = P[i], y = P[i + hp];
        P[i] = add2(x, y);
        P[i + hp] = sub2(x, y);
      }
    }
    // strides 32, 64 across the chunk's lanes: upper = lower - upper
#pragma unroll
    for (int m = 1; m < 4; m <<= 1) {
      const float sg = (a4 & m) ? -1.f : 1.f;
      const uint64_t SG = pk2(sg, sg);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float lo, hi;
        upk2(P[i], lo, hi);
        const uint64_t O = pk2(__shfl_xor_sync(0xffffffffu, lo, m), __shfl_xor_sync(0xffffffffu, hi, m));
        P[i] = fma2(SG, P[i], O);  // o + v (lower) or o - v (upper), exact sign
      }
    }
    if constexpr (TQ) {
      // y = d2 RN(t c) on pairs; the lane's partial sum of squares in index
      // order; the smallest |y| (the bound of the fast quotient)
      const uint64_t C2 = pk2(hadamard_scale(), hadamard_scale());
      uint64_t Y[16];
      float ss = 0.f, ymin = INFINITY;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint64_t V = mul2(P[i], C2);
        float lo, hi, q0, q1;
        upk2(V, lo, hi);
        upk2(mul2(V, V), q0, q1);
        ss = __fadd_rn(__fadd_rn(ss, q0), q1);
        ymin = fminf(ymin, fminf(fabsf(lo), fabsf(hi)));
        lo = __uint_as_float(__float_as_uint(lo) ^ ((d2w << (31 - 2 * i)) & 0x80000000u));
        hi = __uint_as_float(__float_as_uint(hi) ^ ((d2w << (30 - 2 * i)) & 0x80000000u));
        Y[i] = pk2(lo, hi);
      }
      ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, 1));
      ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, 2));
      if (j >= n_tok) continue;  // the shuffles above are done
      const __half n16 = __float2half_rn(fminf(__fsqrt_rn(ss), 65504.0f));
      const float nf = __half2float(n16);
      // magnitude clamps of the lookup: keys k0 and k0 + kTbqBins - 1
      const float alo = __uint_as_float((uint32_t)k0 << 20), ahi = __uint_as_float((uint32_t)(k0 + kTbqBins - 1) << 20);
      auto index = [&](float u) -> uint32_t {
        const uint32_t ub = __float_as_uint(u);
        const int key = (int)(__float_as_uint(fminf(fmaxf(fabsf(u), alo), ahi)) >> 20);
        const float2 e = tbin[key - k0 + (int)(ub >> 31) * kTbqBins];
        return (uint32_t)__float_as_int(e.y) + (u > e.x ? 1u : 0u);
      };
      uint32_t w[4] = {0, 0, 0, 0};
      if (nf == 0.f || (nf < 65504.f && ymin >= 0x1p-100f)) {
        const float r = nf == 0.f ? 0.f : __frcp_rn(nf);
        const uint64_t R2 = pk2(r, r), NN2 = pk2(-nf, -nf);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint64_t Q0 = mul2(Y[i], R2);
          float u0, u1;
          upk2(fma2(fma2(Q0, NN2, Y[i]), R2, Q0), u0, u1);
          w[i >> 2] |= index(u0) << (8 * (i & 3)) | index(u1) << (8 * (i & 3) + 4);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float y0, y1;
          upk2(Y[i], y0, y1);
          const float u0 = nf > 0.f ? __fdiv_rn(y0, nf) : 0.f, u1 = nf > 0.f ? __fdiv_rn(y1, nf) : 0.f;
          w[i >> 2] |= index(u0) << (8 * (i & 3)) | index(u1) << (8 * (i & 3) + 4);
        }
      }
      uint8_t* blk = out + j * ROW + chunk * BB;
      if (a4 == 0) *reinterpret_cast<__half*>(blk) = n16;
      uint16_t* p = reinterpret_cast<uint16_t*>(blk + 2 + 16 * a4);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        p[2 * k] = (uint16_t)w[k];
        p[2 * k + 1] = (uint16_t)(w[k] >> 16);
      }
      continue;
    }
    float v[32];
    float mt = 0.f;  // max |t|
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      upk2(P[i], v[2 * i], v[2 * i + 1]);
      mt = fmaxf(mt, fmaxf(fabsf(v[2 * i]), fabsf(v[2 * i + 1])));
    }
    float mx = __fmul_rn(mt, hadamard_scale());  // max |RN(t c)|
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    if (j >= n_tok) continue;  // the shuffles above are done

    const __half s16 = block_scale_of(mx, qmax);
    const float sf = __half2float(s16);
    const float rcp = sf == 0.f ? 0.f : __frcp_rn(sf);
    const bool clamp = !(sf >= kMinNormalF16 && sf < 65504.f);  // subnormal or saturated scale
    const float lim = clamp ? __fmul_rn((float)qmax, sf) : INFINITY;
    uint32_t w[B];
    const float crc = __fmul_rn(hadamard_scale(), rcp);
    if (clamp || rot_codes_packed<B>(P, crc, w) > kNearHalf) {
      auto f = [&](int) { return crc; };
      auto g = [&](int) { return hadamard_scale(); };
      rot_codes<B, true>(v, f, g, lim, sf, w);
    }
    // d2: negate the fields of the flipped values (a carry may cross a word
    // inside a 3-bit field, never out of one)
    if constexpr (B == 4) {
#pragma unroll
      for (int k = 0; k < 4; ++k) w[k] = (w[k] ^ negx[k]) + negl[k];
    } else {
      const uint32_t x0 = w[0] ^ negx[0], x1 = w[1] ^ negx[1], x2 = w[2] ^ negx[2];
      asm("add.cc.u32 %0, %3, %6;\n\taddc.cc.u32 %1, %4, %7;\n\taddc.u32 %2, %5, %8;"
          : "=r"(w[0]), "=r"(w[1]), "=r"(w[2])
          : "r"(x0), "r"(x1), "r"(x2), "r"(negl[0]), "r"(negl[1]), "r"(negl[2]));
    }
    uint8_t* blk = out + j * ROW + chunk * BB;
    if (a4 == 0) *reinterpret_cast<__half*>(blk) = s16;
    uint16_t* p = reinterpret_cast<uint16_t*>(blk + 2 + 4 * B * a4);
#pragma unroll
    for (int k = 0; k < B; ++k) {
      p[2 * k] = (uint16_t)w[k];
      p[2 * k + 1] = (uint16_t)(w[k] >> 16);
    }
  }
  __syncthreads();
  if (!lo.paged) {
    bool bad = false;
    uint8_t* dst = main_row(lo, a.cp, which, layer, seq, h, u0, &bad);
    if (span_ok(lo, a.cp, which, dst, (int64_t)n_tok * ROW)) copy_out_any(dst, out, n_tok * ROW);
    return;
  }
  // paged: the tile's page ids are read once, in parallel; then one warp per
  // page copies that page's run of rows (16-bit words: rows start at even
  // offsets, 32-bit words when both ends allow)
  __shared__ int pid[kRotItem / 16 + 2];
  const int p0 = u0 / lo.pt, np = (u1 - 1) / lo.pt - p0 + 1;  // pt >= 16: np <= kRotItem / 16 + 1
  if (threadIdx.x < np) pid[threadIdx.x] = a.cp.block_table[(int64_t)seq * lo.max_pages + p0 + threadIdx.x];
  __syncthreads();
  for (int pi = warp; pi < np; pi += kAppendThreads / 32) {
    const int page = pid[pi];
    if (page < 0 || page >= lo.n_pages) {
      if (lane == 0) page_bad = 1;
      continue;
    }
    const int ta = max(u0, (p0 + pi) * lo.pt), tb = min(u1, (p0 + pi + 1) * lo.pt);
    uint8_t* dst = (which ? a.cp.v_main : a.cp.k_main) +
                   ((((int64_t)layer * lo.n_pages + page) * lo.H + h) * lo.pt + ta % lo.pt) * ROW;
    const uint8_t* src = out + (ta - u0) * ROW;
    const int bytes = (tb - ta) * ROW;
    if (!span_ok(lo, a.cp, which, dst, bytes)) continue;  // bounds-checked build only
    const uintptr_t al = reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src) | (uintptr_t)bytes;
    if ((al & 15u) == 0) {  // whole pages: 16 rows of 66 or 50 bytes are whole 16-byte words
      for (int e = lane; e < bytes / 16; e += 32)
        reinterpret_cast<uint4*>(dst)[e] = reinterpret_cast<const uint4*>(src)[e];
    } else if ((al & 3u) == 0) {
      for (int e = lane; e < bytes / 4; e += 32)
        reinterpret_cast<uint32_t*>(dst)[e] = reinterpret_cast<const uint32_t*>(src)[e];
    } else {
      for (int e = lane; e < bytes / 2; e += 32)
        reinterpret_cast<uint16_t*>(dst)[e] = reinterpret_cast<const uint16_t*>(src)[e];
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && page_bad) atomicOr(a.status, KVQ_DEV_PAGE);
}

template <int NC, int DT, int B, bool TQ = false>
void launch_rot(const AppendArgs& a, int which, cudaStream_t st) {
  const int chunks = (a.max_new + kRotItem - 1) / kRotItem + 2;
  const dim3 grid(chunks, a.lo.H, a.n_layers * a.lo.B);
  if (which == 0) quant_rot128_kernel<NC, DT, B, 0, TQ><<<grid, kAppendThreads, 0, st>>>(a);
  else quant_rot128_kernel<NC, DT, B, 1, TQ><<<grid, kAppendThreads, 0, st>>>(a);
}

template <int NC, int DT>
bool rot_tensor(const AppendArgs& a, int which, bool dry, cudaStream_t st) {
  const FmtInfo& f = fmt_main(a.lo, which);
  if (f.codebook) return dry || (launch_rot<NC, DT, 4, true>(a, which, st), true);
  if (f.bits == 4) return dry || (launch_rot<NC, DT, 4>(a, which, st), true);
  if (f.bits == 3) return dry || (launch_rot<NC, DT, 3>(a, which, st), true);
  return false;
}

}  // namespace

bool launch_fast_rot(const AppendArgs& a, int which, bool dry, cudaStream_t st) {
  const Layout& lo = a.lo;
  const FmtInfo& f = fmt_main(lo, which);
  if (lo.tiered || f.axis != KVQ_AXIS_TOKEN || f.group != 128 || f.zp) return false;
  if (lo.paged && lo.pt < 16) return false;  // the page-id cache holds kRotItem / 16 + 2 entries
  if (lo.dtype == KVQ_DT_F16)
    return lo.D == 128 ? rot_tensor<1, KVQ_DT_F16>(a, which, dry, st) : rot_tensor<2, KVQ_DT_F16>(a, which, dry, st);
  return lo.D == 128 ? rot_tensor<1, KVQ_DT_BF16>(a, which, dry, st) : rot_tensor<2, KVQ_DT_BF16>(a, which, dry, st);
}

}  // namespace kvq
