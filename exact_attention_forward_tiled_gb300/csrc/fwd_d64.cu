// Forward kernel instances for head dimension 64 (2 query tile(s) of 128 rows
// per work tile, 8 K/V ring slots).
#include "fwd_kernel.cuh"

namespace fa {
cudaError_t launch_fwd_d64(const FwdLaunch& L) { return launch_fwd_impl<64, 2, 8>(L); }
}  // namespace fa
