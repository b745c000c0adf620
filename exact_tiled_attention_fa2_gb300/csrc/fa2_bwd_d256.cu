// Backward kernels for head dim 256: a CTA per (128-key tile, half of d),
// 64-row query tiles, one CTA per SM.
#include "fa2_bwd256.cuh"

namespace fa2 {
int launch_bwd_d256(const BwdLaunchArgs& a) {
  return a.bf16 ? launch_bwd256_dtype<true>(a) : launch_bwd256_dtype<false>(a);
}
}  // namespace fa2
