// The split-K combine of decode attention (trefon.com "Matematyka cache KV",
// "Jak 4-bitowemu cache to uchodzi": the decode splits the cached tokens and
// merges the pieces' softmax states).  Split s of a (layer, sequence, kv
// head) unit leaves, per query head, its running maximum m_s and sum l_s of
// 2^(score - m_s) (log2 domain) and its unnormalized output O_s; the merge is
// M = max_s m_s, w_s = 2^(m_s - M), L = sum_s w_s l_s, O = sum_s w_s O_s / L.
#pragma once

#include "kvq_internal.cuh"

namespace kvq {

// Floats per (unit, split, query head) partial row: O[0, D), then m, l and
// two pad floats, so that every O row starts 16-byte aligned.
KVQ_HD constexpr int part_row(int D) { return D + 4; }

// The merge of n partial rows of one unit (row i at base + i * step rows of
// [g] query heads), run by one CTA (all NTHREADS threads).  A warp per query
// head reduces m and l over the rows (lanes over rows) and leaves the
// weights w_i in shared memory (wsm: g * n floats, lsm: g floats, 2 g for a
// partial output, which keeps M there too); then every
// thread sums four channels of O at a time over the rows with 16-byte loads,
// eight rows at a time.
// FINAL: the normalized output O / L into dst [g][D]; otherwise one partial
// row (O unnormalized, M, L) into dst [g][part_row], which may be row 0 of
// the input (every element is read before it is written, by the thread that
// writes it).  Partials are read with ld.global.cg (written by other CTAs of
// this launch).
template <int D, int NTHREADS, bool FINAL>
__device__ __forceinline__ void combine_rows(float* base, int n, int step, int g, float* dst, float* wsm,
                                             float* lsm) {
  constexpr int R = part_row(D), NW = NTHREADS / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rstride = (int64_t)step * g * R;  // floats between consecutive merged rows
  float* msm = lsm + g;                           // [g]: M per query head (partial output only)
  for (int hh = warp; hh < g; hh += NW) {
    float M = -INFINITY;
    for (int s = lane; s < n; s += 32) M = fmaxf(M, __ldcg(base + s * rstride + (int64_t)hh * R + D));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f;
    for (int s = lane; s < n; s += 32) {
      const float* p = base + s * rstride + (int64_t)hh * R + D;
      const float w = M == -INFINITY ? 0.f : exp2f(__ldcg(p) - M);
      wsm[hh * n + s] = w;
      L += w * __ldcg(p + 1);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (lane == 0) {
      lsm[hh] = L;
      if constexpr (!FINAL) msm[hh] = M;
    }
  }
  __syncthreads();
  const float4* b4 = reinterpret_cast<const float4*>(base);
  const int64_t stride = rstride / 4;  // float4s between merged rows
  for (int e = threadIdx.x; e < g * (D / 4); e += NTHREADS) {
    const int hh = e / (D / 4), d4 = e % (D / 4);
    const float* w = wsm + hh * n;
    const float4* p = b4 + (int64_t)hh * (R / 4) + d4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int s = 0;
    for (; s + 8 <= n; s += 8) {  // eight rows' loads in flight
      float4 v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = __ldcg(p + (s + k) * stride);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float wk = w[s + k];
        acc.x = fmaf(wk, v[k].x, acc.x);
        acc.y = fmaf(wk, v[k].y, acc.y);
        acc.z = fmaf(wk, v[k].z, acc.z);
        acc.w = fmaf(wk, v[k].w, acc.w);
      }
    }
    for (; s < n; ++s) {
      const float4 v = __ldcg(p + s * stride);
      const float wk = w[s];
      acc.x = fmaf(wk, v.x, acc.x);
      acc.y = fmaf(wk, v.y, acc.y);
      acc.z = fmaf(wk, v.z, acc.z);
      acc.w = fmaf(wk, v.w, acc.w);
    }
    if constexpr (FINAL) {
      const float L = lsm[hh];
      float* o = dst + hh * D + 4 * d4;
      o[0] = L > 0.f ? acc.x / L : 0.f;
      o[1] = L > 0.f ? acc.y / L : 0.f;
      o[2] = L > 0.f ? acc.z / L : 0.f;
      o[3] = L > 0.f ? acc.w / L : 0.f;
    } else {
      reinterpret_cast<float4*>(dst + (int64_t)hh * R)[d4] = acc;
    }
  }
  if constexpr (!FINAL) {
    for (int hh = threadIdx.x; hh < g; hh += NTHREADS) {
      dst[(int64_t)hh * R + D] = msm[hh];
      dst[(int64_t)hh * R + D + 1] = lsm[hh];
    }
  }
}

// The merge of one unit's `splits` consecutive partial rows into obuf [g][D].
template <int D, int NTHREADS>
__device__ __forceinline__ void combine_splits(float* base, int splits, int g, float* obuf, float* wsm, float* lsm) {
  combine_rows<D, NTHREADS, true>(base, splits, 1, g, obuf, wsm, lsm);
}

}  // namespace kvq
