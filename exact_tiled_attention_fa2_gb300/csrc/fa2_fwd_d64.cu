// Forward kernel instantiations for head dim 64: two 128-row query tiles per
// CTA sharing each 128-row key/value tile.
#include "fa2_fwd_pingpong.cuh"

namespace fa2 {
int launch_fwd_d64(const LaunchArgs& a) { return launch_fwd_pingpong_dispatch<64>(a); }
}  // namespace fa2
