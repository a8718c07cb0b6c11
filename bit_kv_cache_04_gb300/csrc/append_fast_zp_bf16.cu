// Specialized phase B of quantize-on-append for asymmetric (scale + zero
// point) 32-value blocks, bf16 input (compiled with --fmad=false).
#include "append_fast.cuh"

namespace kvq {

bool launch_fast_zp_bf16(const AppendArgs& a, int which, bool dry, cudaStream_t st) {
  return a.lo.D == 128 ? launch_fast_zp_tensor<1, KVQ_DT_BF16>(a, which, dry, st)
                       : launch_fast_zp_tensor<2, KVQ_DT_BF16>(a, which, dry, st);
}

}  // namespace kvq
