// Fused decode step kernels (decode_mma.cuh with the step's append) for KIVI-4 caches (symmetric or asymmetric blocks).
#include <type_traits>

#include "decode_mma.cuh"

namespace kvq {

// Fused-step layouts of this file: launches (unless `dry`) into *err; false
// when the cache is not one of them.
bool step_fused_kivi(const DecodeArgs& a, cudaStream_t st, bool dry, cudaError_t* err) {
  const Layout& lo = a.lo;
  if (!mma_layout_ok(lo) || lo.kf.codebook || lo.D != 128 || lo.g > 4) return false;
  const bool rot = (lo.flags & (KVQ_ROTATE_K | KVQ_ROTATE_V)) != 0;
  const bool rope = (lo.flags & KVQ_K_PRE_ROPE) != 0;
  const int TOK = KVQ_AXIS_TOKEN, CH = KVQ_AXIS_CHANNEL;
  const FmtInfo &k = lo.kf, &v = lo.vf;
  auto run = [&](auto cfg, auto step) {
    if (!dry) *err = launch_mma<decltype(cfg), decltype(step)::value>(a, st);
    return true;
  };
  using S1 = std::integral_constant<int, 1>;  // unrotated formats
  const bool kivi4 = fmt_is(k, 4, 32, CH) && fmt_is(v, 4, 32, TOK);
  if (!kivi4 || rot || rope || lo.tiered) return false;
  if (k.zp) return run(Cfg<128, 1, T_<128, KF_CH4, 32, VF_T4, 32, true>, T_<128, KF_CH4, 32, VF_T4, 32, true>, false,
                           false>{}, S1{});
  return run(Cfg<128, 1, T_<128, KF_CH4, 32, VF_T4, 32>, T_<128, KF_CH4, 32, VF_T4, 32>, false, false>{}, S1{});
}

}  // namespace kvq
