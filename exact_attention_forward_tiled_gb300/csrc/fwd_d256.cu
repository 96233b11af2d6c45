// Forward kernel instances for head dimension 256 (1 query tile(s) of 128 rows
// per work tile, 2 K/V ring slots).
#include "fwd_kernel.cuh"

namespace fa {
cudaError_t launch_fwd_d256(const FwdLaunch& L) { return launch_fwd_impl<256, 1, 2>(L); }
}  // namespace fa
