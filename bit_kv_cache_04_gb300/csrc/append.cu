// Quantize-on-append launches (compiled with --fmad=false: the quantizer must
// keep the format's fp32 op order bit for bit; the phase bodies are in
// append_generic.cuh).
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
#include <algorithm>

#include "append_generic.cuh"

namespace kvq {
namespace {

template <int NC, bool ROT>
__global__ void __launch_bounds__(kAppendThreads, 4) append_quantize_kernel(AppendArgs a) {
  extern __shared__ __align__(16) uint8_t sm[];
  append_quantize_unit<NC, ROT>(a, blockIdx.z / a.lo.B, blockIdx.z % a.lo.B, blockIdx.y, blockIdx.x, sm);
}

template <int NC>
__global__ void __launch_bounds__(kAppendThreads) append_requant_kernel(AppendArgs a) {
  append_requant_unit<NC>(a, blockIdx.z / a.lo.B, blockIdx.z % a.lo.B, blockIdx.y, blockIdx.x);
}

__global__ void __launch_bounds__(kAppendThreads) append_window_kernel(AppendArgs a) {
  append_window_unit(a, blockIdx.z / a.lo.B, blockIdx.z % a.lo.B, blockIdx.y, blockIdx.x);
}

__global__ void commit_lengths_kernel(const int32_t* cu_new, int32_t* seq_lens, int batch) {
  int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < batch) seq_lens[b] += cu_new[b + 1] - cu_new[b];
}

}  // namespace

template <int NC, bool ROT>
cudaError_t launch_append_nc(const AppendArgs& a, cudaStream_t st) {
  const Layout& lo = a.lo;
  const int chunks = (a.max_new + kTile - 1) / kTile + 2;
  dim3 grid(chunks, lo.H, a.n_layers * lo.B);
  const size_t smem = 2 * kTile * (lo.D + 8) * sizeof(uint16_t) + (ROT ? 2 * kTile * (lo.D + 1) * sizeof(float) : 0);
  static bool attr_done = false;
  if (!attr_done) {
    cudaFuncSetAttribute(append_quantize_kernel<NC, ROT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 100 * 1024);
    attr_done = true;
  }
  if (lo.tiered) append_requant_kernel<NC><<<grid, kAppendThreads, 0, st>>>(a);
  if (!launch_fast_quantize(a, st)) append_quantize_kernel<NC, ROT><<<grid, kAppendThreads, smem, st>>>(a);
  if (lo.ring) {
    const int wchunks = (std::min(a.max_new, lo.ring) + kTile - 1) / kTile;
    append_window_kernel<<<dim3(wchunks, lo.H, a.n_layers * lo.B), kAppendThreads, 0, st>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_append(const AppendArgs& a, cudaStream_t st) {
  if (a.max_new == 0) return cudaSuccess;
  const bool rot = (a.lo.flags & (KVQ_ROTATE_K | KVQ_ROTATE_V)) != 0;
  if (a.lo.D == 128) return rot ? launch_append_nc<1, true>(a, st) : launch_append_nc<1, false>(a, st);
  return rot ? launch_append_nc<2, true>(a, st) : launch_append_nc<2, false>(a, st);
}

cudaError_t launch_commit_lengths(const int32_t* cu_new, int32_t* seq_lens, int batch, cudaStream_t st) {
  commit_lengths_kernel<<<(batch + 127) / 128, 128, 0, st>>>(cu_new, seq_lens, batch);
  return cudaGetLastError();
}

}  // namespace kvq
