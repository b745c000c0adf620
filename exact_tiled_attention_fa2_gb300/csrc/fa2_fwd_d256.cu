// Forward kernel instantiations for head dim 256 (key tile 64 rows).
#include "fa2_fwd_kernel.cuh"

namespace fa2 {
int launch_fwd_d256(const LaunchArgs& a) { return launch_fwd_dispatch<256, 64>(a); }
}  // namespace fa2
