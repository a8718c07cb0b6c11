// Fused decode step: the tensor-core decode kernel with the append of the
// step's token done by the blocks that own the tiles it changes
// (decode_mma.cuh).  One launch per call for the layouts the step files
// instantiate; false for the others (the caller runs append, then decode).
#include "kvq_internal.cuh"

namespace kvq {

bool step_fused_kivi(const DecodeArgs& a, cudaStream_t st, bool dry, cudaError_t* err);
bool step_fused_d128(const DecodeArgs& a, cudaStream_t st, bool dry, cudaError_t* err);
bool step_fused_d256(const DecodeArgs& a, cudaStream_t st, bool dry, cudaError_t* err);

bool launch_decode_step_fused(const DecodeArgs& a, cudaStream_t st, bool dry, cudaError_t* err) {
  return step_fused_kivi(a, st, dry, err) || step_fused_d128(a, st, dry, err) || step_fused_d256(a, st, dry, err);
}

}  // namespace kvq
