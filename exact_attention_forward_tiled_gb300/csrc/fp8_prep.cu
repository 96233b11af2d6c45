// FP8 preparation of the attention inputs ("FlashAttention-3 (lukebest wiki)",
// technique 3, precision): incoherent processing Q' = QM, K' = KM with
// M = diag(sigma) H_D / sqrt(D) (Hadamard x random signs, orthogonal, so
// Q'K'^T = QK^T), then block quantisation to e4m3 with one fp32 scale per
// 128-row block of each (sequence, head): scale = amax / 448 (1 for an
// all-zero block), code = e4m3(x / scale), round to nearest even, saturating.
//
// One CTA owns one 128 x D block of one tensor. Warp w holds rows
// [w * RPW, (w + 1) * RPW) of the block; lane l holds the D/32 consecutive
// elements d = l * VPL ... of each row, so a row is one coalesced 2*D-byte
// load and one D-byte store. The Walsh-Hadamard transform runs in registers:
// butterflies over the bits of d inside a lane, then across lanes with
// shuffles. The block amax is reduced in shared memory before any code is
// written, so each element is read from HBM once.
#include <cstdint>
#include <cuda_fp16.h>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

struct PrepBatch {
  PrepParams t[3];
  int count[3];  // CTAs (blocks) of each tensor
  int n;
};

template <int D>
__device__ __forceinline__ void load_row(const PrepParams& P, int64_t off, float (&x)[D / 32]) {
  constexpr int VPL = D / 32;
  const uint16_t* src = reinterpret_cast<const uint16_t*>(P.x) + off;
  uint16_t h[VPL];
  if constexpr (VPL == 2) {
    const uint32_t u = __ldg(reinterpret_cast<const unsigned int*>(src));
    h[0] = u & 0xffffu;
    h[1] = u >> 16;
  } else if constexpr (VPL == 4) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(src));
    h[0] = u.x & 0xffffu; h[1] = u.x >> 16; h[2] = u.y & 0xffffu; h[3] = u.y >> 16;
  } else {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(src));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      h[2 * k] = w[k] & 0xffffu;
      h[2 * k + 1] = w[k] >> 16;
    }
  }
#pragma unroll
  for (int j = 0; j < VPL; ++j)
    x[j] = P.bf16 ? __uint_as_float((uint32_t)h[j] << 16) : __half2float(__ushort_as_half(h[j]));
}

template <int D>
__global__ void __launch_bounds__(32 * (D / 16)) fp8_prep_kernel(const PrepBatch pb) {
  constexpr int NW = D / 16;        // warps per CTA
  constexpr int RPW = 128 / NW;     // rows per warp
  constexpr int VPL = D / 32;       // elements per lane per row
  constexpr int LOG_VPL = VPL == 2 ? 1 : (VPL == 4 ? 2 : 3);
  constexpr int LOG_D = LOG_VPL + 5;
  __shared__ float red[NW];

  int bid = blockIdx.x, ti = 0;
  while (ti < pb.n - 1 && bid >= pb.count[ti]) {
    bid -= pb.count[ti];
    ++ti;
  }
  const PrepParams& P = pb.t[ti];
  const int blk = bid % P.nblk;
  const int bh = bid / P.nblk;
  const int h = bh % P.H, b = bh / P.H;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  float sg[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) sg[j] = P.sigma ? (float)P.sigma[lane * VPL + j] : 1.f;
  const float norm = P.sigma ? rsqrtf((float)D) : 1.f;

  float x[RPW][VPL];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    const int row = blk * 128 + warp * RPW + i;
    if (row < P.S) {
      load_row<D>(P, (((int64_t)b * P.S + row) * P.H + h) * D + lane * VPL, x[i]);
    } else {
#pragma unroll
      for (int j = 0; j < VPL; ++j) x[i][j] = 0.f;
    }
    if (P.sigma) {
#pragma unroll
      for (int j = 0; j < VPL; ++j) x[i][j] *= sg[j];
      // butterflies over the bits of d held inside the lane
#pragma unroll
      for (int bit = 0; bit < LOG_VPL; ++bit) {
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
          if (j & (1 << bit)) continue;
          const float a = x[i][j], c = x[i][j | (1 << bit)];
          x[i][j] = a + c;
          x[i][j | (1 << bit)] = a - c;
        }
      }
      // butterflies over the bits of d that select the lane
#pragma unroll
      for (int bit = LOG_VPL; bit < LOG_D; ++bit) {
        const int m = 1 << (bit - LOG_VPL);
        const bool upper = lane & m;
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
          const float other = __shfl_xor_sync(0xffffffffu, x[i][j], m);
          x[i][j] = upper ? other - x[i][j] : x[i][j] + other;
        }
      }
#pragma unroll
      for (int j = 0; j < VPL; ++j) x[i][j] *= norm;
    }
#pragma unroll
    for (int j = 0; j < VPL; ++j) amax = fmaxf(amax, fabsf(x[i][j]));
  }
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) amax = fmaxf(amax, red[w]);
  const float scale = amax > 0.f ? amax / 448.f : 1.f;
  const float inv = 1.f / scale;
  if (threadIdx.x == 0) P.scale[(int64_t)bh * P.nblk + blk] = scale;

#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    const int row = blk * 128 + warp * RPW + i;
    if (row >= P.S) continue;
    uint8_t* dst = P.x8 + (((int64_t)b * P.S + row) * P.H + h) * D + lane * VPL;
    uint32_t w[VPL / 2];
#pragma unroll
    for (int j = 0; j < VPL / 2; ++j) w[j] = ptx::pack_e4m3x2(x[i][2 * j] * inv, x[i][2 * j + 1] * inv);
    if constexpr (VPL == 2) {
      *reinterpret_cast<uint16_t*>(dst) = (uint16_t)w[0];
    } else if constexpr (VPL == 4) {
      *reinterpret_cast<uint32_t*>(dst) = w[0] | (w[1] << 16);
    } else {
      *reinterpret_cast<uint2*>(dst) = make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
    }
  }
}

cudaError_t launch_fp8_prep(const PrepParams* tensors, int n_tensors, int D, cudaStream_t stream) {
  PrepBatch pb{};
  long total = 0;
  pb.n = n_tensors;
  for (int i = 0; i < n_tensors; ++i) {
    pb.t[i] = tensors[i];
    pb.count[i] = tensors[i].B * tensors[i].H * tensors[i].nblk;
    total += pb.count[i];
  }
  if (total == 0) return cudaSuccess;
  if (total > 0x7fffffffL) return cudaErrorInvalidValue;
  switch (D) {
    case 64: fp8_prep_kernel<64><<<(unsigned)total, 32 * 4, 0, stream>>>(pb); break;
    case 128: fp8_prep_kernel<128><<<(unsigned)total, 32 * 8, 0, stream>>>(pb); break;
    case 256: fp8_prep_kernel<256><<<(unsigned)total, 32 * 16, 0, stream>>>(pb); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace fa
