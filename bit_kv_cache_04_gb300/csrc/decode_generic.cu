// Split-K decode attention, generic path: every tier and format.
//
// Grid (split, kv head, layer x sequence); each CTA walks a contiguous range
// of 32-token tiles of one (layer, sequence, kv head), dequantizes each tile
// into shared memory (fp32, in the stored domain: rotated for rotated
// formats, RoPE applied on the fly to keys stored pre-RoPE), scores it for
// the H_q/H_kv query heads that share the kv head, and keeps an online
// softmax (m, l, acc) per head.  The last CTA of a (layer, sequence, kv head)
// to finish (an atomic ticket, nobody waits) merges the split partials and
// undoes the value rotation once (trefon.com "Matematyka cache KV",
// "najpierw obrot": rotate the query once, read blocks as code x scale, rotate
// the output back once).  Scores follow nalar.dev "Kuantisasi KV Cache...":
// s_i = q.k_i / sqrt(D), output = sum_i p_i v_i.
#include "block_codec.cuh"
#include "split_combine.cuh"

namespace kvq {
namespace {

constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

struct TileRef {
  int seg;  // 0 cold, 1 main/hot, 2 window
  int t0, n;
};

__device__ __forceinline__ TileRef tile_at(int tile, int n_c, int n_m, int ce, int qe, int T) {
  TileRef r;
  if (tile < n_c) {
    r.seg = 0;
    r.t0 = tile * kTile;
    r.n = kTile;
  } else if (tile < n_c + n_m) {
    r.seg = 1;
    r.t0 = ce + (tile - n_c) * kTile;
    r.n = min(kTile, qe - r.t0);
  } else {
    r.seg = 2;
    r.t0 = qe + (tile - n_c - n_m) * kTile;
    r.n = min(kTile, T - r.t0);
  }
  return r;
}

// Dequantizes tokens [t0, t0 + n) of one (layer, seq, kv head) into
// x[j * ld + d] in the stored domain.
__device__ void load_tile(const Layout& lo, const CachePtrs& cp, int which, int layer, int seq, int h,
                          const TileRef& tr, float* x, int ld, uint32_t* bad_page) {
  const int D = lo.D;
  if (tr.seg == 2) {
    for (int e = threadIdx.x; e < tr.n * D; e += blockDim.x) {
      const int j = e / D, d = e % D;
      x[j * ld + d] = in_to_f32(resid_row(lo, cp, which, layer, seq, h, tr.t0 + j)[d], lo.dtype);
    }
    return;
  }
  const FmtInfo& f = tr.seg == 0 ? fmt_cold(lo, which) : fmt_main(lo, which);
  if (f.axis == KVQ_AXIS_CHANNEL) {
    bool bad = false;
    const uint8_t* row = tr.seg == 0 ? cold_row(lo, cp, which, layer, seq, h, tr.t0)
                                     : main_row(lo, cp, which, layer, seq, h, tr.t0, &bad);
    for (int c = threadIdx.x; c < D; c += blockDim.x)
      if (f.zp) dequant_zp_serial(row + (int64_t)c * f.bb, f.group, f.bits, x + c, ld);
      else dequant_block_serial(row + (int64_t)c * f.bb, f.group, f.bits, x + c, ld);
    return;
  }
  const int nb = D / f.group;
  for (int item = threadIdx.x; item < tr.n * nb; item += blockDim.x) {
    const int j = item / nb, b = item % nb;
    bool bad = false;
    const uint8_t* row = tr.seg == 0 ? cold_row(lo, cp, which, layer, seq, h, tr.t0 + j)
                                     : main_row(lo, cp, which, layer, seq, h, tr.t0 + j, &bad);
    float* dst = x + j * ld + b * f.group;
    if (bad) {
      *bad_page = 1;
      for (int i = 0; i < f.group; ++i) dst[i] = 0.0f;
      continue;
    }
    if (f.codebook) dequant_tbq4_serial(row + (int64_t)b * f.bb, lo.cb, dst, 1);
    else if (f.zp) dequant_zp_serial(row + (int64_t)b * f.bb, f.group, f.bits, dst, 1);
    else dequant_block_serial(row + (int64_t)b * f.bb, f.group, f.bits, dst, 1);
  }
}

// Rotates rows [0, n) of x (stride ld) in place, 128-chunk by 128-chunk.
__device__ void rotate_rows(float* x, int ld, int n, int D, const uint32_t* d1, const uint32_t* d2, bool inverse) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int chunks = D / 128;
  for (int r = warp; r < n * chunks; r += nw) {
    float* p = x + (r / chunks) * ld + (r % chunks) * 128 + 4 * lane;
    float v[4] = {p[0], p[1], p[2], p[3]};
    if (inverse)
      warp_unrotate128(v, d1, d2);
    else
      warp_rotate128(v, d1, d2);
    p[0] = v[0];
    p[1] = v[1];
    p[2] = v[2];
    p[3] = v[3];
  }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int D>
__global__ void __launch_bounds__(kThreads) decode_generic_kernel(DecodeArgs a) {
  // programmatic dependent launch: see launch_dependent
  grid_dependency_wait();
  grid_launch_dependents();
  constexpr int LD = D + 1;
  constexpr int R = (kMaxGqa * D + kThreads - 1) / kThreads;
  extern __shared__ float sm[];
  float* ks = sm;                  // [kTile][LD]
  float* vs = ks + kTile * LD;     // [kTile][LD]
  float* qs = vs + kTile * LD;     // [g][D], log2-domain scaled
  float* ps = qs + kMaxGqa * D;    // [g][kTile]
  __shared__ float m_s[kMaxGqa], l_s[kMaxGqa], alpha_s[kMaxGqa];
  __shared__ uint32_t bad_page;
  __shared__ int is_last;

  const Layout& lo = a.lo;
  const int g = lo.g;
  const int split = blockIdx.x, h = blockIdx.y;
  const int li = blockIdx.z / lo.B, seq = blockIdx.z % lo.B;
  const int layer = a.layer0 + li;
  const int tid = threadIdx.x;

  int T = a.seq_lens[seq] + a.len_add;
  if (T < 0 || T > lo.max_T) {
    if (split == 0 && h == 0 && tid == 0) atomicOr(a.status, KVQ_DEV_LENGTH);
    T = 0;
  }
  const int qe = q_end_of(lo, T), ce = c_end_of(lo, T);
  const int n_c = ce / kTile;
  const int n_m = (qe - ce + kTile - 1) / kTile;
  const int n_w = (T - qe + kTile - 1) / kTile;
  const int ntiles = n_c + n_m + n_w;
  const int tb = (int)((int64_t)split * ntiles / a.splits);
  const int te = (int)((int64_t)(split + 1) * ntiles / a.splits);

  // query prep: fp32, rotated when K is stored rotated, scaled by log2(e)/sqrt(D)
  const int64_t qrow = ((int64_t)li * lo.B + seq) * lo.Hq + (int64_t)h * g;
  for (int e = tid; e < g * D; e += kThreads) qs[e] = in_to_f32(a.q[qrow * D + e], lo.dtype);
  if (tid < kMaxGqa) {
    m_s[tid] = -INFINITY;
    l_s[tid] = 0.0f;
  }
  if (tid == 0) bad_page = 0;
  __syncthreads();
  if (lo.flags & KVQ_ROTATE_K) {
    rotate_rows(qs, D, g, D, lo.d1, lo.d2, false);
    __syncthreads();
  }
  const float qscale = kLog2e / sqrtf((float)D);
  for (int e = tid; e < g * D; e += kThreads) qs[e] *= qscale;

  float acc[R];
#pragma unroll
  for (int r = 0; r < R; ++r) acc[r] = 0.0f;

  const bool pre_rope = (lo.flags & KVQ_K_PRE_ROPE) != 0;
  const float2* rope_off = a.rope + (int64_t)a.rope_base_rows * (D / 2);

  for (int tile = tb; tile < te; ++tile) {
    const TileRef tr = tile_at(tile, n_c, n_m, ce, qe, T);
    __syncthreads();
    load_tile(lo, a.cp, 0, layer, seq, h, tr, ks, LD, &bad_page);
    load_tile(lo, a.cp, 1, layer, seq, h, tr, vs, LD, &bad_page);
    __syncthreads();
    if (tr.seg == 2 && (lo.flags & (KVQ_ROTATE_K | KVQ_ROTATE_V))) {
      // window tokens are stored unrotated: bring them into the rotated domain
      if (lo.flags & KVQ_ROTATE_K) rotate_rows(ks, LD, tr.n, D, lo.d1, lo.d2, false);
      if (lo.flags & KVQ_ROTATE_V) rotate_rows(vs, LD, tr.n, D, lo.d1, lo.d2, false);
      __syncthreads();
    }
    if (pre_rope) {
      for (int e = tid; e < tr.n * (D / 2); e += kThreads) {
        const int j = e / (D / 2), i = e % (D / 2), t = tr.t0 + j;
        const float2 b = a.rope[(int64_t)(t / kTile) * (D / 2) + i];
        const float2 o = rope_off[(t % kTile) * (D / 2) + i];
        const float c = b.x * o.x - b.y * o.y;
        const float s = b.y * o.x + b.x * o.y;
        float* kr = ks + j * LD;
        const float x0 = kr[i], x1 = kr[i + D / 2];
        kr[i] = x0 * c - x1 * s;
        kr[i + D / 2] = x0 * s + x1 * c;
      }
      __syncthreads();
    }
    // scores and online softmax: warp hh = query head, lane = token
    if (tid < g * 32) {
      const int hh = tid >> 5, j = tid & 31;
      float s = -INFINITY;
      if (j < tr.n) {
        const float* kr = ks + j * LD;
        const float* qr = qs + hh * D;
        float dot = 0.0f;
#pragma unroll 8
        for (int d = 0; d < D; ++d) dot += qr[d] * kr[d];
        s = dot;
      }
      const float m_old = m_s[hh];
      const float m_new = fmaxf(m_old, warp_max(s));
      const float p = j < tr.n ? exp2f(s - m_new) : 0.0f;
      const float sum = warp_sum(p);
      ps[hh * kTile + j] = p;
      __syncwarp();
      if (j == 0) {
        const float alpha = exp2f(m_old - m_new);
        alpha_s[hh] = alpha;
        l_s[hh] = l_s[hh] * alpha + sum;
        m_s[hh] = m_new;
      }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int pidx = tid + r * kThreads;
      const int hh = pidx / D, d = pidx % D;
      if (hh < g) {
        float v = acc[r] * alpha_s[hh];
        const float* pr = ps + hh * kTile;
        for (int j = 0; j < tr.n; ++j) v += pr[j] * vs[j * LD + d];
        acc[r] = v;
      }
    }
  }
  __syncthreads();
  if (tid == 0 && bad_page) atomicOr(a.status, KVQ_DEV_PAGE);

  float* obuf = ks;  // [g][D] final outputs
  const int64_t unit = ((int64_t)li * lo.B + seq) * lo.H + h;
  if (a.splits == 1) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int pidx = tid + r * kThreads;
      const int hh = pidx / D, d = pidx % D;
      if (hh < g) obuf[hh * D + d] = l_s[hh] > 0.0f ? acc[r] / l_s[hh] : 0.0f;
    }
  } else {
    constexpr int PR = part_row(D);
    float* part = a.partials + (unit * a.splits + split) * (int64_t)g * PR;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int pidx = tid + r * kThreads;
      const int hh = pidx / D, d = pidx % D;
      if (hh < g) part[hh * PR + d] = acc[r];
    }
    if (tid < g) {
      part[tid * PR + D] = m_s[tid];
      part[tid * PR + D + 1] = l_s[tid];
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      const unsigned ticket = atomicAdd(a.tickets + unit, 1u);
      is_last = ticket == (unsigned)(a.splits - 1);
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    // the V tile is dead here: the merge weights use it
    static_assert(kTile * LD >= kMaxGqa * kMaxSplits, "merge weights fit in the V tile");
    combine_splits<D, kThreads>(a.partials + unit * a.splits * (int64_t)g * PR, a.splits, g, obuf, vs, l_s);
    if (tid == 0) a.tickets[unit] = 0;
  }
  __syncthreads();
  if (lo.flags & KVQ_ROTATE_V) {
    rotate_rows(obuf, D, g, D, lo.d1, lo.d2, true);
    __syncthreads();
  }
  for (int e = tid; e < g * D; e += kThreads) a.out[qrow * D + e] = obuf[e];
}

template <int D>
cudaError_t launch_generic(const DecodeArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(float) * (2 * kTile * (D + 1) + kMaxGqa * D + kMaxGqa * kTile);
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(decode_generic_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  dim3 grid(a.splits, a.lo.H, a.n_layers * a.lo.B);
  return launch_dependent(decode_generic_kernel<D>, grid, dim3(kThreads), smem, st, a);
}

}  // namespace

cudaError_t launch_decode_generic(const DecodeArgs& a, cudaStream_t st) {
  if (a.lo.D == 128) return launch_generic<128>(a, st);
  return launch_generic<256>(a, st);
}

}  // namespace kvq
