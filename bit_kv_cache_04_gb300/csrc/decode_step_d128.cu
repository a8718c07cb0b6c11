// Fused decode step kernels (decode_mma.cuh with the step's append) for D = 128: KIVI hot/cold tiers with pre-RoPE keys and 66 B / 128 blocks.
#include <type_traits>

#include "decode_mma.cuh"

namespace kvq {

// Fused-step layouts of this file: launches (unless `dry`) into *err; false
// when the cache is not one of them.
bool step_fused_d128(const DecodeArgs& a, cudaStream_t st, bool dry, cudaError_t* err) {
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
  using S2 = std::integral_constant<int, 2>;  // rotated formats
  if (k.zp) return false;
  if (lo.tiered) {  // KIVI-4 hot, KIVI-2 cold, pre-RoPE keys
    if (!rope || rot || !fmt_is(k, 4, 32, CH) || !fmt_is(v, 4, 32, TOK) || !fmt_is(lo.kc, 2, 32, CH) ||
        !fmt_is(lo.vc, 2, 32, TOK))
      return false;
    return run(Cfg<128, 1, T_<128, KF_CH4, 32, VF_T4, 32>, T_<128, KF_CH2, 32, VF_T2, 32>, true, true>{}, S1{});
  }
  // 66 B / 128, rotated or not, no window
  if (rope || lo.ring || !fmt_is(k, 4, 128, TOK) || !fmt_is(v, 4, 128, TOK)) return false;
  return run(Cfg<128, 1, T_<128, KF_T4, 128, VF_T4, 128>, T_<128, KF_T4, 128, VF_T4, 128>, false, false>{}, S2{});
  return false;
}

}  // namespace kvq
