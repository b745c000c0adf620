// Backward kernel instantiations for head dim 64.
#include "fa2_bwd.cuh"

namespace fa2 {
int launch_bwd_d64(const BwdLaunchArgs& a) { return launch_bwd_dispatch<64>(a); }
}  // namespace fa2
