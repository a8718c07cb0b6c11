// Fused decode step kernels (decode_mma.cuh with the step's append) for D = 256: 66 B / 128 and 50 B / 128 blocks.
#include <type_traits>

#include "decode_mma.cuh"

namespace kvq {

// Fused-step layouts of this file: launches (unless `dry`) into *err; false
// when the cache is not one of them.
bool step_fused_d256(const DecodeArgs& a, cudaStream_t st, bool dry, cudaError_t* err) {
  const Layout& lo = a.lo;
  if (!mma_layout_ok(lo) || lo.kf.codebook || lo.D != 256 || lo.g > 8) return false;
  const bool rope = (lo.flags & KVQ_K_PRE_ROPE) != 0;
  const int TOK = KVQ_AXIS_TOKEN;
  const FmtInfo &k = lo.kf, &v = lo.vf;
  auto run = [&](auto cfg, auto step) {
    if (!dry) *err = launch_mma<decltype(cfg), decltype(step)::value>(a, st);
    return true;
  };
  using S2 = std::integral_constant<int, 2>;  // rotated formats
  if (k.zp || lo.tiered || rope || lo.ring) return false;
  if (fmt_is(k, 4, 128, TOK) && fmt_is(v, 4, 128, TOK))
    return run(Cfg<256, 1, T_<256, KF_T4, 128, VF_T4, 128>, T_<256, KF_T4, 128, VF_T4, 128>, false, false, true>{}, S2{});
  if (fmt_is(k, 3, 128, TOK) && fmt_is(v, 3, 128, TOK))
    return run(Cfg<256, 1, T_<256, KF_T3, 128, VF_T3, 128>, T_<256, KF_T3, 128, VF_T3, 128>, false, false, true>{}, S2{});
  return false;
}

}  // namespace kvq
