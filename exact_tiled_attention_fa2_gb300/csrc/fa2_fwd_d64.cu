// Forward kernel instantiations for head dim 64 (key tile 128 rows).
#include "fa2_fwd_kernel.cuh"

namespace fa2 {
int launch_fwd_d64(const LaunchArgs& a) { return launch_fwd_dispatch<64, 128>(a); }
}  // namespace fa2
