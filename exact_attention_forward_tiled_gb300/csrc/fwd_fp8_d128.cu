// e4m3 forward kernel instances for head dimension 128 (2 query tiles of 128
// rows per work tile, 10 K/V ring slots of 16 KB).
#include "fwd_kernel.cuh"

namespace fa {
cudaError_t launch_fwd_fp8_d128(const FwdLaunch& L) { return launch_fwd_kind<128, 2, 10, kE4M3>(L); }
}  // namespace fa
