// e4m3 forward kernel instances for head dimension 64 (2 query tiles of 128
// rows per work tile; a 64-byte row is one box in the 64-byte swizzle;
// 16 K/V ring slots of 8 KB).
#include "fwd_kernel.cuh"

namespace fa {
cudaError_t launch_fwd_fp8_d64(const FwdLaunch& L) { return launch_fwd_kind<64, 2, 16, kE4M3>(L); }
}  // namespace fa
