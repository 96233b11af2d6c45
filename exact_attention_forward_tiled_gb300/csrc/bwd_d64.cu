// Backward kernels, head dimension 64: 8 streamed tiles in flight (16 KB each).
#include "bwd_kernel.cuh"

namespace fa {
cudaError_t launch_bwd_d64(const BwdLaunch& L) { return launch_bwd_impl<64, 8, 8>(L); }
}  // namespace fa
