// Specialized phase B of quantize-on-append (compiled with --fmad=false like
// the generic kernels): 32-value blocks of unrotated formats with symmetric
// codes, and the dispatch of every specialized format.
#include "append_fast.cuh"

namespace kvq {
namespace {

// Launches the specialized phase B of tensor `which` when one exists for its
// format; false otherwise (nothing launched).
template <int NC, int DT>
bool launch_fast_tensor(const AppendArgs& a, int which, bool dry, cudaStream_t st) {
  const Layout& lo = a.lo;
  const FmtInfo& f = fmt_main(lo, which);
  const bool rot = (lo.flags & (which ? KVQ_ROTATE_V : KVQ_ROTATE_K)) != 0;
  if (rot) return launch_fast_rot(a, which, dry, st);  // Hadamard formats: their own translation unit
  if (f.group != 32) return false;
  const int cb = lo.tiered ? fmt_cold(lo, which).bits : 0;
  if (f.zp) {  // asymmetric blocks (4- or 2-bit, 4 -> 2 tiers): their own translation units
    return DT == KVQ_DT_F16 ? launch_fast_zp_f16(a, which, dry, st) : launch_fast_zp_bf16(a, which, dry, st);
  }
  if (f.axis == KVQ_AXIS_CHANNEL) {  // keys (values grouped per channel take the generic kernel)
    if (which != 0) return false;
    if (f.bits == 4 && cb == 0) return dry || (launch_channel32<NC, DT, 4, 0>(a, st), true);
    if (f.bits == 4 && cb == 2) return dry || (launch_channel32<NC, DT, 4, 2>(a, st), true);
    if (f.bits == 2 && cb == 0) return dry || (launch_channel32<NC, DT, 2, 0>(a, st), true);
    return false;
  }
  if (cb == 0) {
    switch (f.bits) {
      case 8: return dry || (launch_token32<NC, DT, 8, 0>(a, which, st), true);
      case 4: return dry || (launch_token32<NC, DT, 4, 0>(a, which, st), true);
      case 3: return dry || (launch_token32<NC, DT, 3, 0>(a, which, st), true);
      case 2: return dry || (launch_token32<NC, DT, 2, 0>(a, which, st), true);
    }
    return false;
  }
  if (f.bits == 4 && cb == 2 && which == 1) return dry || (launch_token32<NC, DT, 4, 2>(a, which, st), true);
  return false;
}

template <int NC>
bool launch_fast_nc(const AppendArgs& a, cudaStream_t st) {
  if (a.lo.dtype == KVQ_DT_F16) {
    if (!launch_fast_tensor<NC, KVQ_DT_F16>(a, 0, true, st) || !launch_fast_tensor<NC, KVQ_DT_F16>(a, 1, true, st))
      return false;
    launch_fast_tensor<NC, KVQ_DT_F16>(a, 0, false, st);
    launch_fast_tensor<NC, KVQ_DT_F16>(a, 1, false, st);
    return true;
  }
  if (!launch_fast_tensor<NC, KVQ_DT_BF16>(a, 0, true, st) || !launch_fast_tensor<NC, KVQ_DT_BF16>(a, 1, true, st))
    return false;
  launch_fast_tensor<NC, KVQ_DT_BF16>(a, 0, false, st);
  launch_fast_tensor<NC, KVQ_DT_BF16>(a, 1, false, st);
  return true;
}

}  // namespace

bool launch_fast_quantize(const AppendArgs& a, cudaStream_t st) {
  return a.lo.D == 128 ? launch_fast_nc<1>(a, st) : launch_fast_nc<2>(a, st);
}

bool fast_quantize_available(const AppendArgs& a) {
  if (a.lo.dtype == KVQ_DT_F16)
    return a.lo.D == 128 ? launch_fast_tensor<1, KVQ_DT_F16>(a, 0, true, 0) && launch_fast_tensor<1, KVQ_DT_F16>(a, 1, true, 0)
                         : launch_fast_tensor<2, KVQ_DT_F16>(a, 0, true, 0) && launch_fast_tensor<2, KVQ_DT_F16>(a, 1, true, 0);
  return a.lo.D == 128 ? launch_fast_tensor<1, KVQ_DT_BF16>(a, 0, true, 0) && launch_fast_tensor<1, KVQ_DT_BF16>(a, 1, true, 0)
                       : launch_fast_tensor<2, KVQ_DT_BF16>(a, 0, true, 0) && launch_fast_tensor<2, KVQ_DT_BF16>(a, 1, true, 0);
}

}  // namespace kvq
