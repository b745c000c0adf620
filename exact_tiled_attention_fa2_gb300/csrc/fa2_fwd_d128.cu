// Forward kernel instantiations for head dim 128: two 128-row query tiles per
// CTA sharing each 128-row key/value tile.
#include "fa2_fwd_pingpong.cuh"

namespace fa2 {
int launch_fwd_d128(const LaunchArgs& a) { return launch_fwd_pingpong_dispatch<128>(a); }
}  // namespace fa2
