// Pieces shared by the append translation units (generic and specialized
// phase B): block size, the span of one sequence's append, input rows.
#pragma once

#include "block_codec.cuh"

namespace kvq {
namespace {

constexpr int kAppendThreads = 128;

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(sa), "l"(gmem));
}
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
  const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(sa), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

struct SeqSpan {
  int T0, T1, n, off;
  bool ok;
};

__device__ __forceinline__ SeqSpan read_span(const AppendArgs& a, int seq) {
  SeqSpan s;
  if (a.one_per_seq) {
    s.off = seq;
    s.n = 1;
  } else {
    s.off = a.cu_new[seq];
    s.n = a.cu_new[seq + 1] - s.off;
  }
  s.T0 = a.seq_lens[seq];
  s.T1 = s.T0 + s.n;
  uint32_t bad = 0;
  if (s.n < 0 || s.T0 < 0 || s.T0 > a.lo.max_T || s.off < 0 || s.off + s.n > a.total_new) bad |= KVQ_DEV_LENGTH;
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

}  // namespace
}  // namespace kvq
