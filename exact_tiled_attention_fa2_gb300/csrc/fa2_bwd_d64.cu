// Backward kernels for head dim 64: 64-row query tiles, two CTAs per SM.
#include "fa2_bwd64.cuh"

namespace fa2 {
int launch_bwd_d64(const BwdLaunchArgs& a) {
  return a.bf16 ? launch_bwd64_dtype<true>(a) : launch_bwd64_dtype<false>(a);
}
}  // namespace fa2
