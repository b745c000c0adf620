// Backward kernel instantiations for head dim 128.
#include "fa2_bwd.cuh"

namespace fa2 {
int launch_bwd_d128(const BwdLaunchArgs& a) { return launch_bwd_dispatch<128>(a); }
}  // namespace fa2
