// Backward kernels, head dimension 128: 4 streamed tiles in flight (32 KB each).
#include "bwd_kernel.cuh"

namespace fa {
cudaError_t launch_bwd_d128(const BwdLaunch& L) { return launch_bwd_impl<128, 4>(L); }
}  // namespace fa
