// Backward kernels, head dimension 128: 4 streamed tiles in flight (32 KB
// each) in the dK/dV kernel, 5 in the dQ kernel (which needs no per-warp
// column constants, so a fifth tile fits in shared memory).
#include "bwd_kernel.cuh"

namespace fa {
cudaError_t launch_bwd_d128(const BwdLaunch& L) { return launch_bwd_impl<128, 4, 5>(L); }
}  // namespace fa
