// Per-row constants of the attention backward, one pass over O and dO:
//   delta[h][t] = sum_d dO[t, h, d] * O[t, h, d]   (= sum_j P_tj dP_tj, the
//                 softmax-Jacobian term of row t)
//   lse2[h][t]  = LSE[t, h] * log2(e), +inf where LSE = -inf (a row that sees
//                 no key: every recomputed P of it is then exp2(-inf) = 0)
// A (token, head) row is spread over D / 8 lanes holding 8 consecutive
// elements each (16-byte loads); the dot product is finished with shuffles.
#include <cstdint>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "fa_internal.h"

namespace fa {
namespace {

__device__ __forceinline__ float to_f(uint16_t u, bool fp16) {
  return fp16 ? __half2float(__ushort_as_half(u)) : __uint_as_float((uint32_t)u << 16);
}

template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const uint16_t* __restrict__ o,
                                                       const uint16_t* __restrict__ dout,
                                                       const float* __restrict__ lse, float* __restrict__ lse2,
                                                       float* __restrict__ delta, int total_q, int H, int Sq,
                                                       int lse_varlen, int fp16) {
  constexpr int LPR = D / 8;
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t row = gid / LPR;          // t * H + h
  const int part = (int)(gid % LPR);
  const bool in = row < (int64_t)total_q * H;
  float acc = 0.f;
  if (in) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(o + row * D + part * 8));
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(dout + row * D + part * 8));
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      acc = fmaf(to_f(wa[k] & 0xffffu, fp16), to_f(wb[k] & 0xffffu, fp16), acc);
      acc = fmaf(to_f(wa[k] >> 16, fp16), to_f(wb[k] >> 16, fp16), acc);
    }
  }
#pragma unroll
  for (int m = LPR / 2; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
  if (in && part == 0) {
    const int t = (int)(row / H), h = (int)(row % H);
    const int64_t li = lse_varlen ? (int64_t)h * total_q + t : ((int64_t)(t / Sq) * H + h) * Sq + t % Sq;
    const float l = lse[li];
    const int64_t out = (int64_t)h * total_q + t;
    lse2[out] = l == -CUDART_INF_F ? CUDART_INF_F : l * 1.4426950408889634f;
    delta[out] = acc;
  }
}

}  // namespace

cudaError_t launch_bwd_prep(const void* o, const void* dout, const float* lse, float* lse2, float* delta,
                            int total_q, int H, int D, int Sq, int lse_varlen, int fp16, cudaStream_t stream) {
  const int64_t threads = (int64_t)total_q * H * (D / 8);
  if (threads == 0) return cudaSuccess;
  const int64_t blocks = (threads + 255) / 256;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  const auto* po = static_cast<const uint16_t*>(o);
  const auto* pd = static_cast<const uint16_t*>(dout);
  if (D == 64)
    bwd_prep_kernel<64><<<(unsigned)blocks, 256, 0, stream>>>(po, pd, lse, lse2, delta, total_q, H, Sq, lse_varlen, fp16);
  else if (D == 128)
    bwd_prep_kernel<128><<<(unsigned)blocks, 256, 0, stream>>>(po, pd, lse, lse2, delta, total_q, H, Sq, lse_varlen, fp16);
  else if (D == 256)
    bwd_prep_kernel<256><<<(unsigned)blocks, 256, 0, stream>>>(po, pd, lse, lse2, delta, total_q, H, Sq, lse_varlen, fp16);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace fa
