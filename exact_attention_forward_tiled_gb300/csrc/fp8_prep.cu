// FP8 preparation of the attention inputs ("FlashAttention-3 (lukebest wiki)",
// technique 3, precision): incoherent processing Q' = QM, K' = KM with
// M = diag(sigma) H_D / sqrt(D) (Hadamard x random signs, orthogonal, so
// Q'K'^T = QK^T), then block quantisation to e4m3 with one fp32 scale per
// 128-row block of each (sequence, head): scale = amax / 448 (1 for an
// all-zero block), code = e4m3(x / scale), round to nearest even, saturating.
//
// One CTA owns one 128 x D block of one tensor and keeps it in registers:
// the Walsh-Hadamard transform runs there (butterflies over the bits of d
// inside a lane, then across lanes with shuffles), the block amax is reduced
// through shared memory, and only then are the codes written, so every
// element is read from HBM once and written once.
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

// Eight consecutive 16-bit elements (16 bytes) -> fp32.
__device__ __forceinline__ void load8(const PrepParams& P, int64_t off, float (&x)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(P.x) + off));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint16_t lo = w[k] & 0xffffu, hi = w[k] >> 16;
    x[2 * k] = P.bf16 ? __uint_as_float((uint32_t)lo << 16) : __half2float(__ushort_as_half(lo));
    x[2 * k + 1] = P.bf16 ? __uint_as_float((uint32_t)hi << 16) : __half2float(__ushort_as_half(hi));
  }
}

// CTA = one 128-row block of one (sequence, head) of one tensor. A row is
// spread over LPR = D/8 lanes holding 8 consecutive elements each (16-byte
// loads, 8-byte stores), so one warp instruction covers 32/LPR rows.
// Consecutive CTAs take consecutive heads of the same rows, so the CTAs in
// flight read whole [token, H*D] rows of HBM.
template <int D>
__global__ void __launch_bounds__(32 * (D == 256 ? 32 : 16), D == 256 ? 1 : 2) fp8_prep_kernel(const PrepBatch pb) {
  constexpr int NW = D == 256 ? 32 : 16;  // warps per CTA (4 loads in flight per lane)
  constexpr int LPR = D / 8;               // lanes per row
  constexpr int RPI = 32 / LPR;            // rows per warp instruction
  constexpr int RPW = 128 / NW;            // rows per warp
  constexpr int ITER = RPW / RPI;
  constexpr int LOG_D = D == 64 ? 6 : (D == 128 ? 7 : 8);
  __shared__ float red[NW];

  int bid = blockIdx.x, ti = 0;
  while (ti < pb.n - 1 && bid >= pb.count[ti]) {
    bid -= pb.count[ti];
    ++ti;
  }
  const PrepParams& P = pb.t[ti];
  const int h = bid % P.H;
  const int rest = bid / P.H;
  const int b = rest % P.B;
  const int blk = rest / P.B;
  // the block's rows: tokens start + [blk * 128, min(blk * 128 + 128, L))
  int64_t start = (int64_t)b * P.S;
  int L = P.S;
  int64_t sidx = ((int64_t)b * P.H + h) * P.nblk + blk;   // where its scale goes
  if (P.cu_seqlens != nullptr) {
    const int s0 = __ldg(P.cu_seqlens + b), s1 = __ldg(P.cu_seqlens + b + 1);
    const int c0 = __ldg(P.cu_blocks + b), c1 = __ldg(P.cu_blocks + b + 1), cn = __ldg(P.cu_blocks + P.B);
    // bad lengths, or block offsets that do not span exactly this sequence's
    // blocks within the first cu_blocks[B] <= total / 128 + B rows of the
    // [n_blocks, H] scale arrays: skipped and reported
    if (s0 < 0 || s1 < s0 || s1 > P.total || s1 - s0 > P.S || c0 < 0 || c1 - c0 != (s1 - s0 + 127) / 128 ||
        c1 > cn || cn > P.total / 128 + P.B) {
      if (threadIdx.x == 0 && blk == 0 && h == 0) atomicOr(P.status, kDevBadSeqlens);
      return;
    }
    start = s0;
    L = s1 - s0;
    if (blk * 128 >= L) return;   // the whole CTA leaves together
    sidx = (int64_t)(c0 + blk) * P.H + h;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane / LPR;              // row of the instruction this lane serves
  const int d0 = (lane % LPR) * 8;         // first element of the lane

  float sg[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) sg[j] = P.sigma ? (float)P.sigma[d0 + j] : 1.f;
  // 1/sqrt(D) of the rotation is applied once, in the quantisation multiplier
  const float norm = P.sigma ? rsqrtf((float)D) : 1.f;

  float x[ITER][8];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < ITER; ++i) {
    const int row = blk * 128 + warp * RPW + i * RPI + sub;
    if (row < L) {
      load8(P, ((start + row) * P.H + h) * D + d0, x[i]);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) x[i][j] = 0.f;
    }
  }
#pragma unroll
  for (int i = 0; i < ITER; ++i) {
    if (P.sigma) {
#pragma unroll
      for (int j = 0; j < 8; ++j) x[i][j] *= sg[j];
      // Walsh-Hadamard butterflies over the three bits of d inside the lane
#pragma unroll
      for (int bit = 0; bit < 3; ++bit) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (j & (1 << bit)) continue;
          const float a = x[i][j], c = x[i][j | (1 << bit)];
          x[i][j] = a + c;
          x[i][j | (1 << bit)] = a - c;
        }
      }
      // ... and over the bits of d that select the lane (within the row's
      // lanes): lower partner a + b, upper partner a - b = other - mine, one
      // FFMA each with the sign of the lane's half
#pragma unroll
      for (int bit = 3; bit < LOG_D; ++bit) {
        const int m = 1 << (bit - 3);
        const float sgn = (lane & m) ? -1.f : 1.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float other = __shfl_xor_sync(0xffffffffu, x[i][j], m);
          x[i][j] = fmaf(x[i][j], sgn, other);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(x[i][j]));
  }
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) amax = fmaxf(amax, red[w]);
  amax *= norm;   // amax of the rotated, normalised values
  const float scale = amax > 0.f ? amax / 448.f : 1.f;
  const float inv = norm / scale;
  if (threadIdx.x == 0) P.scale[sidx] = scale;

#pragma unroll
  for (int i = 0; i < ITER; ++i) {
    const int row = blk * 128 + warp * RPW + i * RPI + sub;
    if (row >= L) continue;
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) w[j] = ptx::pack_e4m3x2(x[i][2 * j] * inv, x[i][2 * j + 1] * inv);
    *reinterpret_cast<uint2*>(P.x8 + ((start + row) * P.H + h) * D + d0) =
        make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
  }
}

// cu_blocks[b] = sum over b' < b of ceil(L_b' / 128), L_b = cu_seqlens[b+1] - cu_seqlens[b]
// (a negative length counts as 0). One thread: B is small next to the rest.
__global__ void varlen_blocks_kernel(const int* __restrict__ cu_seqlens, int B, int* __restrict__ cu_blocks) {
  if (blockIdx.x != 0 || threadIdx.x != 0) return;
  int acc = 0;
  cu_blocks[0] = 0;
  for (int b = 0; b < B; ++b) {
    const int L = cu_seqlens[b + 1] - cu_seqlens[b];
    acc += L > 0 ? (L + 127) / 128 : 0;
    cu_blocks[b + 1] = acc;
  }
}

cudaError_t launch_varlen_blocks(const int* cu_seqlens, int B, int* cu_blocks, cudaStream_t stream) {
  varlen_blocks_kernel<<<1, 32, 0, stream>>>(cu_seqlens, B, cu_blocks);
  return cudaGetLastError();
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
    case 64: fp8_prep_kernel<64><<<(unsigned)total, 32 * 16, 0, stream>>>(pb); break;
    case 128: fp8_prep_kernel<128><<<(unsigned)total, 32 * 16, 0, stream>>>(pb); break;
    case 256: fp8_prep_kernel<256><<<(unsigned)total, 32 * 32, 0, stream>>>(pb); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace fa
