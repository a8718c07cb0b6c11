// Decode attention: the tensor-core kernel (decode_mma.cuh) when the cache's
// formats fit it, else the generic kernel.
#include "decode_mma.cuh"

namespace kvq {
namespace {

// Launches (unless `dry`) the tensor-core decode kernel for the cache's
// formats into *err; false when none fits.
bool dispatch_mma(const DecodeArgs& a, cudaStream_t st, bool dry, cudaError_t* err) {
  const Layout& lo = a.lo;
  auto run = [&](auto cfg) {
    if (!dry) *err = launch_mma<decltype(cfg), 0>(a, st);
    return true;
  };
  const int TOK = KVQ_AXIS_TOKEN, CH = KVQ_AXIS_CHANNEL;
  const bool rope = (lo.flags & KVQ_K_PRE_ROPE) != 0;
  if (!mma_layout_ok(lo)) return false;
  if (lo.kf.codebook) {  // TBQ4 K and V (rotated 4-bit blocks of 128)
    if (lo.D == 128 && lo.g <= 4)
      return run(Cfg<128, 1, T_<128, KF_TQ, 128, VF_TQ, 128>, T_<128, KF_TQ, 128, VF_TQ, 128>, false, false>{});
    if (lo.D == 256 && lo.g <= 8)
      return run(Cfg<256, 1, T_<256, KF_TQ, 128, VF_TQ, 128>, T_<256, KF_TQ, 128, VF_TQ, 128>, false, false, true>{});
    return false;
  }
  const FmtInfo &k = lo.kf, &v = lo.vf;
  const bool kivi4 = fmt_is(k, 4, 32, CH) && fmt_is(v, 4, 32, TOK);
  using KIVI4 = T_<128, KF_CH4, 32, VF_T4, 32>;
  using KIVI2 = T_<128, KF_CH2, 32, VF_T2, 32>;
  if (k.zp) {  // asymmetric KIVI: per-channel K, per-token V, blocks of 32
    using Z4 = T_<128, KF_CH4, 32, VF_T4, 32, true>;
    using Z2 = T_<128, KF_CH2, 32, VF_T2, 32, true>;
    const bool kivi2 = fmt_is(k, 2, 32, CH) && fmt_is(v, 2, 32, TOK);
    if (lo.D == 128 && lo.g <= 4) {
      if (lo.tiered) {
        if (kivi4 && fmt_is(lo.kc, 2, 32, CH) && fmt_is(lo.vc, 2, 32, TOK)) {
          if (rope) return run(Cfg<128, 1, Z4, Z2, true, true>{});
          return run(Cfg<128, 1, Z4, Z2, true, false>{});
        }
      } else if (kivi4) {
        if (rope) return run(Cfg<128, 1, Z4, Z4, false, true>{});
        return run(Cfg<128, 1, Z4, Z4, false, false>{});
      } else if (kivi2 && !rope) {
        return run(Cfg<128, 1, Z2, Z2, false, false>{});
      }
    }
    return false;
  }
  if (lo.D == 128 && lo.g <= 4 && kivi4) {
    if (lo.tiered) {
      if (fmt_is(lo.kc, 2, 32, CH) && fmt_is(lo.vc, 2, 32, TOK)) {
        if (rope) return run(Cfg<128, 1, KIVI4, KIVI2, true, true>{});
        return run(Cfg<128, 1, KIVI4, KIVI2, true, false>{});
      }
    } else {
      if (rope) return run(Cfg<128, 1, KIVI4, KIVI4, false, true>{});
      return run(Cfg<128, 1, KIVI4, KIVI4, false, false>{});
    }
  }
  if (lo.tiered || rope) return false;
  if (lo.D == 128 && lo.g <= 4) {
    using A = T_<128, KF_T4, 128, VF_T4, 128>;
    using B = T_<128, KF_T4, 32, VF_T4, 32>;
    using Q8 = T_<128, KF_T8, 32, VF_T8, 32>;
    if (fmt_is(k, 4, 128, TOK) && fmt_is(v, 4, 128, TOK)) return run(Cfg<128, 1, A, A, false, false>{});
    if (fmt_is(k, 4, 32, TOK) && fmt_is(v, 4, 32, TOK)) return run(Cfg<128, 1, B, B, false, false>{});
    if (fmt_is(k, 8, 32, TOK) && fmt_is(v, 8, 32, TOK)) return run(Cfg<128, 1, Q8, Q8, false, false>{});
  }
  if (lo.D == 256 && lo.g <= 8) {
    using A4 = T_<256, KF_T4, 128, VF_T4, 128>;
    using A3 = T_<256, KF_T3, 128, VF_T3, 128>;
    if (fmt_is(k, 4, 128, TOK) && fmt_is(v, 4, 128, TOK)) return run(Cfg<256, 1, A4, A4, false, false, true>{});
    if (fmt_is(k, 3, 128, TOK) && fmt_is(v, 3, 128, TOK)) return run(Cfg<256, 1, A3, A3, false, false, true>{});
  }
  return false;
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st) {
  cudaError_t e = cudaSuccess;
  if (dispatch_mma(a, st, false, &e)) return e;
  return launch_decode_generic(a, st);
}

}  // namespace kvq
