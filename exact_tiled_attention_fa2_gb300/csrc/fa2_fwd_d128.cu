// Forward kernel instantiations for head dim 128 (key tile 128 rows).
#include "fa2_fwd_kernel.cuh"

namespace fa2 {
int launch_fwd_d128(const LaunchArgs& a) { return launch_fwd_dispatch<128, 128>(a); }
}  // namespace fa2
