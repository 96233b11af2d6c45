// Forward kernel instances for head dimension 64 with one query tile of 128
// rows per work tile (query sequences of at most 128 rows), 12 K/V ring slots.
#include "fwd_kernel.cuh"

namespace fa {
cudaError_t launch_fwd_d64_q1(const FwdLaunch& L) { return launch_fwd_impl<64, 1, 12>(L); }
}  // namespace fa
