// Merge of split-KV partial results (the partial softmax of FlashDecoding,
// named in the lineage of the FlashAttention-3 wiki). Each key range r of a
// query row gave a self-normalised O_r and LSE_r; the row over all keys is
//
//   LSE = ln sum_r exp(LSE_r),   O = sum_r exp(LSE_r - LSE) O_r
//
// (a range with no visible key has LSE_r = -inf and weight 0; a row with no
// visible key at all gets O = 0, LSE = -inf). HBM-bound: one thread owns four
// consecutive elements of one output row, reads the n_split partial rows with
// 16-byte loads and writes O once.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "fa_internal.h"

namespace fa {

template <bool FP16>
__global__ void __launch_bounds__(256) splitkv_merge_kernel(const float* __restrict__ o_part,
                                                            const float* __restrict__ lse_part, void* o,
                                                            float* lse, int n_split, int B, int H, int Sq,
                                                            int D) {
  const int cpr = D / 4;   // threads per output row
  const int64_t tq = (int64_t)B * Sq;
  const int64_t total = tq * H * cpr;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(idx % cpr);
    const int64_t row = idx / cpr;           // (token, head)
    const int h = (int)(row % H);
    const int64_t tok = row / H;
    const int b = (int)(tok / Sq);
    const int i = (int)(tok - (int64_t)b * Sq);
    const int64_t lse_stride = (int64_t)B * H * Sq;
    const int64_t lse_off = ((int64_t)b * H + h) * Sq + i;
    float m = -CUDART_INF_F;
    for (int s = 0; s < n_split; ++s) m = fmaxf(m, __ldg(lse_part + s * lse_stride + lse_off));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float sum = 0.f;
    if (m != -CUDART_INF_F) {
      const int64_t o_stride = tq * H * D;
      const int64_t o_off = row * D + 4 * c;
      for (int s = 0; s < n_split; ++s) {
        const float ls = __ldg(lse_part + s * lse_stride + lse_off);
        const float wgt = ls == -CUDART_INF_F ? 0.f : expf(ls - m);
        sum += wgt;
        if (wgt != 0.f) {
          const float4 v = __ldg(reinterpret_cast<const float4*>(o_part + s * o_stride + o_off));
          acc.x += wgt * v.x;
          acc.y += wgt * v.y;
          acc.z += wgt * v.z;
          acc.w += wgt * v.w;
        }
      }
      const float inv = 1.f / sum;
      acc.x *= inv;
      acc.y *= inv;
      acc.z *= inv;
      acc.w *= inv;
    }
    uint2 packed;
    if (FP16) {
      const __half2 lo = __floats2half2_rn(acc.x, acc.y), hi = __floats2half2_rn(acc.z, acc.w);
      packed = make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
    } else {
      const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
      packed = make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
    }
    *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(o) + row * D + 4 * c) = packed;
    if (c == 0) lse[lse_off] = m == -CUDART_INF_F ? -CUDART_INF_F : m + logf(sum);
  }
}

cudaError_t launch_splitkv_merge(const float* o_part, const float* lse_part, void* o, float* lse,
                                 int n_split, int B, int H, int Sq, int D, int out_fp16, int num_sms,
                                 cudaStream_t stream) {
  const int64_t total = (int64_t)B * Sq * H * (D / 4);
  if (total == 0) return cudaSuccess;
  // grid-stride: at most 64 blocks of 256 threads per SM
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = (int64_t)(num_sms > 0 ? num_sms : 1) * 64;
  if (blocks > cap) blocks = cap;
  if (out_fp16)
    splitkv_merge_kernel<true><<<(unsigned)blocks, 256, 0, stream>>>(o_part, lse_part, o, lse, n_split, B, H, Sq, D);
  else
    splitkv_merge_kernel<false><<<(unsigned)blocks, 256, 0, stream>>>(o_part, lse_part, o, lse, n_split, B, H, Sq, D);
  return cudaGetLastError();
}

}  // namespace fa
