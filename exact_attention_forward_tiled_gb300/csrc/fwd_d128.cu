// Forward kernel instances for head dimension 128 (2 query tile(s) of 128 rows
// per work tile, 4 K/V ring slots).
#include "fwd_kernel.cuh"

namespace fa {
cudaError_t launch_fwd_d128(const FwdLaunch& L) { return launch_fwd_impl<128, 2, 4>(L); }
}  // namespace fa
