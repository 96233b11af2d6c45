// Test helper: throughput of back-to-back tcgen05.mma (M128 N128 K16, bf16,
// fp32 accumulator in tensor memory) issued by one thread per SM, with the
// operand descriptors built the way the forward kernel builds them. FORM 0:
// A and B from shared memory, B K-major (the QK^T products); FORM 1: A from
// tensor memory, B MN-major (the PV products). One CTA per SM (it holds all
// 512 tensor-memory columns); operands are zeros; the commit wait is bounded
// (2 s, a timeout sets *err). Returns cycles per product.
#include <cstdint>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace {

using namespace fa;

template <int FORM>
__global__ void __launch_bounds__(128, 1) mma_issue_kernel(uint32_t b_off, int n, long long* cycles, int* err) {
  extern __shared__ uint8_t raw[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_holder;
  const uint32_t rbase = ptx::smem_u32(raw);
  const uint32_t base = (rbase + 1023u) & ~1023u;
  uint8_t* sm = raw + (base - rbase);
  for (int i = threadIdx.x; i < 64 * 1024 / 16; i += blockDim.x) reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bar), 1);
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_u32(&tmem_holder), 512);
    ptx::tmem_relinquish();
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_holder;
  constexpr uint32_t idesc_qk = ptx::make_idesc(1u, false, 128, 128);
  constexpr uint32_t idesc_pv = ptx::make_idesc(1u, true, 128, 128);
  const long long t0 = clock64();
  if (warp == 0 && lane == 0) {
    const uint32_t a_addr = base, b_addr = base + b_off;
    for (int g = 0; g < n / 8; ++g) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        if (FORM == 0) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          ptx::mma_f16_ss(tmem, ptx::smem_desc_sw128(a_addr + off, 16, 1024),
                          ptx::smem_desc_sw128(b_addr + off, 16, 1024), idesc_qk, kk > 0 || g > 0);
        } else {
          ptx::mma_f16_ts(tmem, tmem + 256 + kk * 8, ptx::smem_desc_sw128(b_addr + kk * 16 * 128, 16384, 1024),
                          idesc_pv, kk > 0 || g > 0);
        }
      }
    }
    ptx::mma_commit(ptx::smem_u32(&bar));
    const uint64_t w0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(ptx::smem_u32(&bar), 0)) {
      if (ptx::globaltimer_ns() - w0 > 2000000000ull) {
        atomicOr(err, 1);
        break;
      }
    }
  }
  __syncthreads();
  const long long t1 = clock64();
  if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

}  // namespace

extern "C" double mma_issue_cycles(int form, int n, int ctas, long long* cycles, int* err) {
  if (n < 8 || ctas < 1 || ctas > 1024) return -1.0;
  const int smem = 120 * 1024;   // one CTA per SM
  cudaError_t e;
  if (form == 0) {
    e = cudaFuncSetAttribute(mma_issue_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) mma_issue_kernel<0><<<ctas, 128, smem>>>(32768u, n, cycles, err);
  } else {
    e = cudaFuncSetAttribute(mma_issue_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) mma_issue_kernel<1><<<ctas, 128, smem>>>(32768u, n, cycles, err);
  }
  if (e != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) return -2.0;
  long long h[1024];
  if (cudaMemcpy(h, cycles, ctas * sizeof(long long), cudaMemcpyDeviceToHost) != cudaSuccess) return -3.0;
  double mean = 0.0;
  for (int i = 0; i < ctas; ++i) mean += (double)h[i] / ctas;
  return mean / n;
}
