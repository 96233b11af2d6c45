// Backward kernels, head dimension 256: three kernels (dQ; dK; dV), streamed
// tiles in 32 KB halves -- 3 slots for dQ, 2 for dK (which also holds V and
// the per-warp column constants), 4 for dV (which holds K only).
#include "bwd_kernel.cuh"

namespace fa {
cudaError_t launch_bwd_d256(const BwdLaunch& L) {
  if (L.kind == kF16) {
    if (L.dq) return launch_bwd_dir<256, 3, kF16, kBwdDQ>(L);
    return L.part == 1 ? launch_bwd_dir<256, 2, kF16, kBwdDK>(L) : launch_bwd_dir<256, 4, kF16, kBwdDV>(L);
  }
  if (L.dq) return launch_bwd_dir<256, 3, kBF16, kBwdDQ>(L);
  return L.part == 1 ? launch_bwd_dir<256, 2, kBF16, kBwdDK>(L) : launch_bwd_dir<256, 4, kBF16, kBwdDV>(L);
}
}  // namespace fa
