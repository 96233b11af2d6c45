// Test helper: one CTA waits, through the attention kernel's own bounded
// waiter, on an mbarrier that nothing ever arrives at. The wait must give up
// after its time limit, record the timeout in the status word, raise the
// CTA's abort flag and return, leaving the CUDA context usable.
#include <cstdint>
#include "fwd_kernel.cuh"

__global__ void wait_on_nothing(int* status, int* result) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    fa::ptx::mbar_init(fa::ptx::smem_u32(&bar), 1);
    abort_flag = 0;
    fa::ptx::fence_mbar_init();
  }
  __syncthreads();
  const fa::Waiter wt{&abort_flag, status};
  const bool ok = wt.wait_warp(fa::ptx::smem_u32(&bar), 0, 11);
  if (threadIdx.x == 0) {
    result[0] = ok ? 1 : 0;
    result[1] = abort_flag;
  }
}

extern "C" int run_wait_on_nothing(int* status, int* result) {
  wait_on_nothing<<<1, 32>>>(status, result);
  return (int)cudaDeviceSynchronize();
}
