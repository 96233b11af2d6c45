// e4m3 forward kernel instances for head dimension 256 (1 query tile of 128
// rows per work tile, 5 K/V ring slots of 32 KB).
#include "fwd_kernel.cuh"

namespace fa {
cudaError_t launch_fwd_fp8_d256(const FwdLaunch& L) { return launch_fwd_kind<256, 1, 5, kE4M3>(L); }
}  // namespace fa
