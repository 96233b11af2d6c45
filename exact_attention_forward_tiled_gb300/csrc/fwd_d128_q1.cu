// Forward kernel instances for head dimension 128 with one query tile of 128
// rows per work tile (query sequences of at most 128 rows), 6 K/V ring slots.
#include "fwd_kernel.cuh"

namespace fa {
cudaError_t launch_fwd_d128_q1(const FwdLaunch& L) { return launch_fwd_impl<128, 1, 6>(L); }
}  // namespace fa
