// Forward kernel instantiations for head dim 256: one 128-row query tile per
// CTA, 64-row key/value tiles, two S buffers in tensor memory.
#include "fa2_fwd_dbuf.cuh"

namespace fa2 {
int launch_fwd_d256(const LaunchArgs& a) { return launch_fwd_dbuf_dispatch<256>(a); }
}  // namespace fa2
