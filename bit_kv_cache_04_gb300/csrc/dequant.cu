// kvq_dequantize (blocks -> fp32 in the original domain) and the RoPE angle
// tables used by decode for keys stored pre-RoPE.
#include "block_codec.cuh"

namespace kvq {
namespace {

constexpr int kThreads = 128;

// Storage of token t of one (layer, seq, head): its row (window row, or the
// main / cold tier row holding it) and the tier (0 main, 1 cold, 2 window);
// row = nullptr for a page id out of range.
struct TokRow {
  const uint8_t* row;
  int tier;
};

__device__ TokRow token_row(const Layout& lo, const CachePtrs& cp, int which, int layer, int seq, int h, int t,
                            int qe, int ce, bool* bad) {
  if (t >= qe) return {reinterpret_cast<const uint8_t*>(resid_row(lo, cp, which, layer, seq, h, t)), 2};
  if (t < ce) return {cold_row(lo, cp, which, layer, seq, h, t), 1};
  return {main_row(lo, cp, which, layer, seq, h, t, bad), 0};
}

// Value of element d of token t (stored domain), its storage row known.
__device__ __forceinline__ float stored_value(const Layout& lo, const TokRow& r, int which, int t, int d) {
  if (r.tier == 2) return in_to_f32(reinterpret_cast<const uint16_t*>(r.row)[d], lo.dtype);
  if (!r.row) return 0.0f;
  const FmtInfo& f = r.tier == 1 ? fmt_cold(lo, which) : fmt_main(lo, which);
  if (f.axis == KVQ_AXIS_CHANNEL) {
    const uint8_t* blk = r.row + (int64_t)d * f.bb;
    return block_value(blk, f.bits, 0, f.zp, lo.cb, t % f.group);
  }
  const uint8_t* blk = r.row + (int64_t)(d / f.group) * f.bb;
  return block_value(blk, f.bits, f.codebook, f.zp, lo.cb, d % f.group);
}

__global__ void __launch_bounds__(kThreads) dequantize_kernel(DequantArgs a) {
  extern __shared__ float xs[];  // [kTile][D]
  const Layout& lo = a.lo;
  const int D = lo.D, h = blockIdx.y;
  const int T = a.seq_lens[a.seq];
  if (T < 0 || T > lo.max_T || a.t1 > T) {
    if (blockIdx.x == 0 && h == 0 && threadIdx.x == 0) atomicOr(a.status, KVQ_DEV_RANGE);
    return;
  }
  const int qe = q_end_of(lo, T), ce = c_end_of(lo, T);
  const int t0 = a.t0 + blockIdx.x * kTile;
  const int n = min(kTile, a.t1 - t0);
  if (n <= 0) return;
  __shared__ uint32_t bad_page;
  __shared__ TokRow rows[kTile];
  if (threadIdx.x == 0) bad_page = 0;
  for (int which = 0; which < 2; ++which) {
    __syncthreads();
    if (threadIdx.x < n) {  // each token's row once
      bool bad = false;
      rows[threadIdx.x] = token_row(lo, a.cp, which, a.layer, a.seq, h, t0 + threadIdx.x, qe, ce, &bad);
      if (bad) bad_page = 1;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < n * D; e += blockDim.x) {
      const int j = e / D, d = e % D;
      xs[e] = stored_value(lo, rows[j], which, t0 + j, d);
    }
    __syncthreads();
    if (lo.flags & (which ? KVQ_ROTATE_V : KVQ_ROTATE_K)) {
      // quantized tokens are stored rotated: undo it; window tokens are raw
      const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
      for (int r = warp; r < n * (D / 128); r += nw) {
        const int j = r / (D / 128);
        if (t0 + j >= qe) continue;
        float* p = xs + j * D + (r % (D / 128)) * 128 + 4 * lane;
        float v[4] = {p[0], p[1], p[2], p[3]};
        warp_unrotate128(v, lo.d1, lo.d2);
        p[0] = v[0];
        p[1] = v[1];
        p[2] = v[2];
        p[3] = v[3];
      }
      __syncthreads();
    }
    float* out = which ? a.v_out : a.k_out;
    for (int e = threadIdx.x; e < n * D; e += blockDim.x) {
      const int j = e / D, d = e % D;
      out[((int64_t)(t0 + j - a.t0) * lo.H + h) * D + d] = xs[e];
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && bad_page) atomicOr(a.status, KVQ_DEV_PAGE);
}

// base[r][i] = (cos, sin)(32 r theta_i), off[j][i] = (cos, sin)(j theta_i),
// theta_i = theta^(-2i/D), evaluated in fp64 and rounded to fp32; then the
// same off values regrouped in the order the tensor-core decode's lanes read
// them: float4 [D/32 chunk pairs kcp][4 tokens k][2 channel pairs][32 lanes],
// lane (gq, tq) holding token j = 4gq + k and channels c + {0, 4} or
// c + {1, 5}, c = 32 (kcp / 2) + 8 tq + 2 (kcp % 2).
__global__ void rope_tables_kernel(float2* rope, int base_rows, int D, double theta) {
  const int half = D / 2;
  const int plain = (base_rows + kTile) * half;
  const int total = plain + kTile * half;
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < total; e += gridDim.x * blockDim.x) {
    int i;
    double pos;
    if (e < plain) {
      const int r = e / half;
      i = e % half;
      pos = r < base_rows ? (double)r * kTile : (double)(r - base_rows);
    } else {
      const int f2 = e - plain, F = f2 >> 1, hf = f2 & 1;
      const int lane = F & 31, qp = (F >> 5) & 1, k = (F >> 6) & 3, kcp = F >> 8;
      const int q = 2 * qp + hf;
      const int dq = q == 0 ? 0 : q == 1 ? 4 : q == 2 ? 1 : 5;
      i = 32 * (kcp >> 1) + 8 * (lane & 3) + 2 * (kcp & 1) + dq;
      pos = (double)(4 * (lane >> 2) + k);
    }
    const double inv = pow(theta, -2.0 * i / D);
    double s, c;
    sincos(pos * inv, &s, &c);
    if (e < plain) {
      rope[e] = make_float2((float)c, (float)s);
    } else {  // fragment order: per 16 bytes (cos q0, cos q1, sin q0, sin q1)
      const int f2 = e - plain;
      float* rf = reinterpret_cast<float*>(rope + plain);
      rf[4 * (f2 >> 1) + (f2 & 1)] = (float)c;
      rf[4 * (f2 >> 1) + 2 + (f2 & 1)] = (float)s;
    }
  }
}

// x rounded to 8 significant bits (nearest, ties to even), then to fp16:
// exact for |x| >= 2^-17, so that x_hi times any integer code of magnitude at
// most 8 is exact in fp16; smaller values land on fp16's 2^-24 grid.
__device__ __half hi8_of(double x) {
  if (x == 0.0) return __double2half(0.0);
  int e;
  frexp(x, &e);  // x = m 2^e, 0.5 <= |m| < 1
  return __double2half(ldexp(rint(ldexp(x, 8 - e)), e - 8));
}

// The turn table of the tensor-core decode's per-channel keys: cos and sin of
// j theta_i (j = 0..31 the token's offset in its 32-token group), each split
// into an fp16 part with 8 significant bits (hi) and the fp16 rounding of the
// rest (lo), so hi + lo holds about 20 bits and code x hi is exact.  Layout:
// uint4 [D/32 chunk pairs kcp][4 tokens k][2 halves][32 lanes] (a warp's
// load of one half is 512 contiguous bytes): for lane (gq, tq), token
// j = 4 gq + k and channel pairs P0 = (c, c + 4), P1 = (c + 1, c + 5),
// c = 32 (kcp / 2) + 8 tq + 2 (kcp % 2), as fp16 pairs (low half the first
// channel): half 0 = (cos hi P0, cos hi P1, cos lo P0, cos lo P1),
// half 1 = (sin hi P0, sin hi P1, sin lo P0, sin lo P1).
__global__ void rope_hilo_kernel(uint32_t* tab, int D, double theta) {
  const int total = (D / 32) * 4 * 32 * 8;
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < total; e += gridDim.x * blockDim.x) {
    // e = (((kcp * 4 + k) * 2 + half) * 32 + lane) * 4 + word
    const int lane = (e >> 2) & 31, k = (e >> 8) & 3, kcp = e >> 10;
    const int w = 4 * ((e >> 7) & 1) + (e & 3);  // word of the 8 (cos hi, cos hi, cos lo, cos lo, sin ...)
    const int p = w & 1, type = w >> 1;  // type: 0 cos hi, 1 cos lo, 2 sin hi, 3 sin lo
    const int c0 = 32 * (kcp >> 1) + 8 * (lane & 3) + 2 * (kcp & 1) + p;
    const double j = (double)(4 * (lane >> 2) + k);
    uint32_t word = 0;
    for (int half_ = 0; half_ < 2; ++half_) {
      const int i = c0 + 4 * half_;
      double s, c;
      sincos(j * pow(theta, -2.0 * i / D), &s, &c);
      const double x = type < 2 ? c : s;
      const __half hi = hi8_of(x);
      const __half v = (type & 1) ? __double2half(x - (double)__half2float(hi)) : hi;
      word |= (uint32_t)__half_as_ushort(v) << (16 * half_);
    }
    tab[e] = word;
  }
}

}  // namespace

cudaError_t launch_dequantize(const DequantArgs& a, cudaStream_t st) {
  dim3 grid((a.t1 - a.t0 + kTile - 1) / kTile, a.lo.H);
  const size_t smem = sizeof(float) * kTile * a.lo.D;
  dequantize_kernel<<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_rope_tables(float2* rope, int base_rows, int D, float theta, cudaStream_t st) {
  rope_tables_kernel<<<256, 256, 0, st>>>(rope, base_rows, D, (double)theta);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // the fp16 hi / lo table follows the fp32 tables: (base_rows + 2 kTile) rows of D/2 float2
  rope_hilo_kernel<<<(D / 32) * 4 * 32 * 8 / 256, 256, 0, st>>>(
      reinterpret_cast<uint32_t*>(rope + (int64_t)(base_rows + 2 * kTile) * (D / 2)), D, (double)theta);
  return cudaGetLastError();
}

}  // namespace kvq
