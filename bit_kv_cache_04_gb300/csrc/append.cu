// Quantize-on-append (compiled with --fmad=false: the quantizer must keep
// the format's fp32 op order bit for bit).
//
// One append of n tokens to a sequence of T0 tokens (T1 = T0 + n) runs three
// launches in stream order, each over every (layer, sequence, kv head):
//   A  hot groups [c_end(T0), min(c_end(T1), q_end(T0))) requantized to the
//      cold format from their dequantized hot values;
//   B  units [q_end(T0), q_end(T1)) quantized from the window (tokens < T0)
//      or the new input; units below c_end(T1) continue to the cold format
//      through the same hot quantize -> dequantize -> requantize;
//   C  new tokens in [max(T0, q_end(T1)), T1) copied into the window ring.
// A runs before B because B may overwrite hot-ring slots that A reads; B
// before C because C may overwrite window slots that B reads.  Keys are
// grouped per channel over 32-token groups and values per token (troisinh.com
// "KV Cache Quantization", "Tai sao Key va Value lai khac nhau?"); rotated
// formats pass each token's 128-chunks through the randomized Hadamard
// transform first (trefon.com "Matematyka cache KV", "najpierw obrot").
#include "block_codec.cuh"

namespace kvq {
namespace {

constexpr int kAppendThreads = 128;

struct SeqSpan {
  int T0, T1, n, off;
  bool ok;
};

__device__ SeqSpan read_span(const AppendArgs& a, int seq) {
  SeqSpan s;
  s.off = a.cu_new[seq];
  s.n = a.cu_new[seq + 1] - s.off;
  s.T0 = a.seq_lens[seq];
  s.T1 = s.T0 + s.n;
  uint32_t bad = 0;
  if (s.n < 0 || s.T0 < 0 || s.T0 > a.lo.max_T || s.off < 0 || a.cu_new[seq + 1] > a.total_new) bad |= KVQ_DEV_LENGTH;
  else if (s.n > a.max_new || s.T1 > a.lo.max_T) bad |= KVQ_DEV_CAPACITY;
  s.ok = bad == 0;
  if (bad && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) atomicOr(a.status, bad);
  return s;
}

__device__ __forceinline__ const uint16_t* input_row(const AppendArgs& a, int which, int li, const SeqSpan& s,
                                                     int h, int t) {
  const uint16_t* base = which ? a.v : a.k;
  int64_t row = ((int64_t)li * a.total_new + s.off + (t - s.T0)) * a.lo.H + h;
  return base + row * a.lo.D;
}

// Writes one quantized per-token row (or per-channel group row) of values
// x (fp32, smem, row stride ld) to the main tier, or to the cold tier after
// a requantization when to_cold.
__device__ void store_unit(const AppendArgs& a, int which, int layer, int seq, int h, int u0, int n_tok,
                           const float* x, int ld, bool to_cold, uint32_t* page_bad) {
  const Layout& lo = a.lo;
  const FmtInfo& f = fmt_main(lo, which);
  const FmtInfo& fc = fmt_cold(lo, which);
  float deq[128];
  if (f.axis == KVQ_AXIS_CHANNEL) {
    // block c = channel c over the group's 32 tokens (token order)
    for (int c = threadIdx.x; c < lo.D; c += blockDim.x) {
      auto get = [&](int j) { return x[j * ld + c]; };
      if (to_cold) {
        alignas(4) uint8_t tmp[2 + 32];
        quant_block_serial(get, f.group, f.bits, tmp, deq);
        uint8_t* dst = cold_row(lo, a.cp, which, layer, seq, h, u0) + (int64_t)c * fc.bb;
        quant_block_serial([&](int j) { return deq[j]; }, fc.group, fc.bits, dst, nullptr);
      } else {
        bool bad = false;
        uint8_t* row = main_row(lo, a.cp, which, layer, seq, h, u0, &bad);
        quant_block_serial(get, f.group, f.bits, row + (int64_t)c * f.bb, nullptr);
      }
    }
    return;
  }
  const int nb = lo.D / f.group;
  for (int item = threadIdx.x; item < n_tok * nb; item += blockDim.x) {
    const int j = item / nb, b = item % nb;
    const int t = u0 + j;
    const float* xr = x + j * ld + b * f.group;
    auto get = [&](int i) { return xr[i]; };
    if (to_cold) {
      alignas(4) uint8_t tmp[2 + 128];
      quant_block_serial(get, f.group, f.bits, tmp, deq);
      uint8_t* dst = cold_row(lo, a.cp, which, layer, seq, h, t) + (int64_t)b * fc.bb;
      quant_block_serial([&](int i) { return deq[i]; }, fc.group, fc.bits, dst, nullptr);
    } else {
      bool bad = false;
      uint8_t* row = main_row(lo, a.cp, which, layer, seq, h, t, &bad);
      if (bad) {
        *page_bad = 1;
        continue;
      }
      quant_block_serial(get, f.group, f.bits, row + (int64_t)b * f.bb, nullptr);
    }
  }
}

// Phase B: quantize units [q_end(T0), q_end(T1)).
__global__ void __launch_bounds__(kAppendThreads) append_quantize_kernel(AppendArgs a) {
  extern __shared__ float xs[];  // [kTile][D + 1]
  __shared__ uint32_t page_bad;
  const Layout& lo = a.lo;
  const int li = blockIdx.z / lo.B, seq = blockIdx.z % lo.B, h = blockIdx.y;
  const int layer = a.layer0 + li;
  SeqSpan s = read_span(a, seq);
  if (!s.ok) return;
  const int q0 = q_end_of(lo, s.T0), q1 = q_end_of(lo, s.T1), c1 = c_end_of(lo, s.T1);
  const int base = (q0 / kTile) * kTile + blockIdx.x * kTile;
  const int u0 = max(base, q0), u1 = min(base + kTile, q1);
  if (u0 >= u1) return;
  const int n_tok = u1 - u0;
  const int ld = lo.D + 1;
  if (threadIdx.x == 0) page_bad = 0;
  for (int which = 0; which < 2; ++which) {
    __syncthreads();
    // gather the unit's tokens (window ring for old tokens, input for new)
    for (int e = threadIdx.x; e < n_tok * lo.D; e += blockDim.x) {
      const int j = e / lo.D, d = e % lo.D, t = u0 + j;
      const uint16_t* src = t < s.T0 ? resid_row(lo, a.cp, which, layer, seq, h, t) : input_row(a, which, li, s, h, t);
      xs[j * ld + d] = in_to_f32(src[d], lo.dtype);
    }
    __syncthreads();
    const bool rotate = (lo.flags & (which ? KVQ_ROTATE_V : KVQ_ROTATE_K)) != 0;
    if (rotate) {
      const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
      for (int r = warp; r < n_tok * (lo.D / 128); r += nw) {
        float* p = xs + (r / (lo.D / 128)) * ld + (r % (lo.D / 128)) * 128 + 4 * lane;
        float v[4] = {p[0], p[1], p[2], p[3]};
        warp_rotate128(v, lo.d1, lo.d2);
        p[0] = v[0];
        p[1] = v[1];
        p[2] = v[2];
        p[3] = v[3];
      }
      __syncthreads();
    }
    const bool to_cold = lo.tiered && u0 < c1;
    store_unit(a, which, layer, seq, h, u0, n_tok, xs, ld, to_cold, &page_bad);
  }
  __syncthreads();
  if (threadIdx.x == 0 && page_bad) atomicOr(a.status, KVQ_DEV_PAGE);
}

// Phase A: hot units [c_end(T0), min(c_end(T1), q_end(T0))) -> cold.
__global__ void __launch_bounds__(kAppendThreads) append_requant_kernel(AppendArgs a) {
  extern __shared__ float xs[];
  const Layout& lo = a.lo;
  const int li = blockIdx.z / lo.B, seq = blockIdx.z % lo.B, h = blockIdx.y;
  const int layer = a.layer0 + li;
  SeqSpan s = read_span(a, seq);
  if (!s.ok) return;
  const int c0 = c_end_of(lo, s.T0), c1 = c_end_of(lo, s.T1), q0 = q_end_of(lo, s.T0);
  const int stop = min(c1, q0);
  const int u0 = c0 + blockIdx.x * kTile;  // c0 and units are whole groups (Gamma = 32)
  if (u0 >= stop) return;
  const int ld = lo.D + 1;
  for (int which = 0; which < 2; ++which) {
    __syncthreads();
    const FmtInfo& f = fmt_main(lo, which);
    bool bad = false;
    if (f.axis == KVQ_AXIS_CHANNEL) {
      const uint8_t* row = main_row(lo, a.cp, which, layer, seq, h, u0, &bad);
      for (int c = threadIdx.x; c < lo.D; c += blockDim.x)
        dequant_block_serial(row + (int64_t)c * f.bb, f.group, f.bits, xs + c, ld);
    } else {
      const int nb = lo.D / f.group;
      for (int item = threadIdx.x; item < kTile * nb; item += blockDim.x) {
        const int j = item / nb, b = item % nb;
        const uint8_t* row = main_row(lo, a.cp, which, layer, seq, h, u0 + j, &bad);
        dequant_block_serial(row + (int64_t)b * f.bb, f.group, f.bits, xs + j * ld + b * f.group, 1);
      }
    }
    __syncthreads();
    // requantize the exact dequantized values to the cold format
    const FmtInfo& fc = fmt_cold(lo, which);
    if (fc.axis == KVQ_AXIS_CHANNEL) {
      for (int c = threadIdx.x; c < lo.D; c += blockDim.x) {
        uint8_t* dst = cold_row(lo, a.cp, which, layer, seq, h, u0) + (int64_t)c * fc.bb;
        quant_block_serial([&](int j) { return xs[j * ld + c]; }, fc.group, fc.bits, dst, nullptr);
      }
    } else {
      const int nb = lo.D / fc.group;
      for (int item = threadIdx.x; item < kTile * nb; item += blockDim.x) {
        const int j = item / nb, b = item % nb;
        uint8_t* dst = cold_row(lo, a.cp, which, layer, seq, h, u0 + j) + (int64_t)b * fc.bb;
        const float* xr = xs + j * ld + b * fc.group;
        quant_block_serial([&](int i) { return xr[i]; }, fc.group, fc.bits, dst, nullptr);
      }
    }
  }
}

// Phase C: new tokens that stay in the 16-bit window.
__global__ void __launch_bounds__(kAppendThreads) append_window_kernel(AppendArgs a) {
  const Layout& lo = a.lo;
  const int li = blockIdx.z / lo.B, seq = blockIdx.z % lo.B, h = blockIdx.y;
  const int layer = a.layer0 + li;
  SeqSpan s = read_span(a, seq);
  if (!s.ok) return;
  const int w0 = max(s.T0, q_end_of(lo, s.T1));
  const int t0 = s.T0 + blockIdx.x * kTile;
  const int ta = max(t0, w0), tb = min(t0 + kTile, s.T1);
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

__global__ void commit_lengths_kernel(const int32_t* cu_new, int32_t* seq_lens, int batch) {
  int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < batch) seq_lens[b] += cu_new[b + 1] - cu_new[b];
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, cudaStream_t st) {
  const Layout& lo = a.lo;
  if (a.max_new == 0) return cudaSuccess;
  const int chunks = (a.max_new + kTile - 1) / kTile + 2;
  dim3 grid(chunks, lo.H, a.n_layers * lo.B);
  const size_t smem = sizeof(float) * kTile * (lo.D + 1);
  static bool attr_done = false;
  if (!attr_done) {
    cudaFuncSetAttribute(append_quantize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
    cudaFuncSetAttribute(append_requant_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
    attr_done = true;
  }
  if (lo.tiered) append_requant_kernel<<<grid, kAppendThreads, smem, st>>>(a);
  append_quantize_kernel<<<grid, kAppendThreads, smem, st>>>(a);
  if (lo.ring) append_window_kernel<<<grid, kAppendThreads, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_commit_lengths(const int32_t* cu_new, int32_t* seq_lens, int batch, cudaStream_t st) {
  commit_lengths_kernel<<<(batch + 127) / 128, 128, 0, st>>>(cu_new, seq_lens, batch);
  return cudaGetLastError();
}

}  // namespace kvq
