// FP8 preparation of the attention inputs ("FlashAttention-3 (lukebest wiki)",
// technique 3, precision): incoherent processing Q' = QM, K' = KM with
// M = diag(sigma) H_D / sqrt(D) (Hadamard x random signs, orthogonal, so
// Q'K'^T = QK^T), then block quantisation to e4m3 with one fp32 scale per
// 128-row block of each (sequence, head): scale = amax / 448 (1 for an
// all-zero block), code = e4m3(x / scale), round to nearest even, saturating.
//
// Persistent CTAs walk the 128 x D blocks (one head of one tensor each); a
// TMA copy brings the next block into shared memory while the current one is
// rotated in registers, its amax is reduced through shared memory and its
// codes are written, so every element is read from HBM once and written once,
// with reads in flight throughout. For D <= 128 a thread owns a whole row and
// runs its Walsh-Hadamard transform on packed fp32 pairs without any
// cross-lane traffic (fp8_prep_rows_kernel); D = 256 spreads a row over 32
// lanes and finishes the transform with shuffles (fp8_prep_lanes_kernel).
#include <cstdint>
#include <cuda_fp16.h>

#include "fa_internal.h"
#include "pipeline.cuh"
#include "ptx.cuh"

namespace fa {

struct PrepBatch {
  PrepParams t[3];
  int count[3];  // CTAs (blocks) of each tensor
  int n;
};

// Eight consecutive 16-bit elements (16 bytes, read from shared memory) -> fp32.
__device__ __forceinline__ void cvt8(uint4 u, bool bf16, float (&x)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint16_t lo = w[k] & 0xffffu, hi = w[k] >> 16;
    x[2 * k] = bf16 ? __uint_as_float((uint32_t)lo << 16) : __half2float(__ushort_as_half(lo));
    x[2 * k + 1] = bf16 ? __uint_as_float((uint32_t)hi << 16) : __half2float(__ushort_as_half(hi));
  }
}

struct PrepMaps {
  CUtensorMap m[3];
};

// shared-memory block buffers per CTA (NB - 1 blocks fetched ahead)
constexpr int kPrepBuffers = 2;

// Where block `bid` (counted over all tensors of the batch) lives: tensor,
// head, first token, valid rows, scale index; false if the block starts past
// its sequence (varlen) or its sequence breaks its bounds (reported).
struct PrepBlock {
  int ti, h, blk, L;
  int64_t start, sidx;
};

__device__ __forceinline__ bool prep_block(const PrepBatch& pb, int bid, PrepBlock& o) {
  int ti = 0;
  while (ti < pb.n - 1 && bid >= pb.count[ti]) {
    bid -= pb.count[ti];
    ++ti;
  }
  const PrepParams& P = pb.t[ti];
  o.ti = ti;
  o.h = bid % P.H;
  const int rest = bid / P.H;
  const int b = rest % P.B;
  o.blk = rest / P.B;
  o.start = (int64_t)b * P.S;
  o.L = P.S;
  o.sidx = ((int64_t)b * P.H + o.h) * P.nblk + o.blk;
  if (P.cu_seqlens != nullptr) {
    const int s0 = __ldg(P.cu_seqlens + b), s1 = __ldg(P.cu_seqlens + b + 1);
    const int c0 = __ldg(P.cu_blocks + b), c1 = __ldg(P.cu_blocks + b + 1), cn = __ldg(P.cu_blocks + P.B);
    // bad lengths, or block offsets that do not span exactly this sequence's
    // blocks within the first cu_blocks[B] <= total / 128 + B rows of the
    // [n_blocks, H] scale arrays: skipped and reported
    if (s0 < 0 || s1 < s0 || s1 > P.total || s1 - s0 > P.S || c0 < 0 || c1 - c0 != (s1 - s0 + 127) / 128 ||
        c1 > cn || cn > P.total / 128 + P.B) {
      if (threadIdx.x == 0 && o.blk == 0 && o.h == 0) atomicOr(P.status, kDevBadSeqlens);
      return false;
    }
    o.start = s0;
    o.L = s1 - s0;
    if (o.blk * 128 >= o.L) return false;
    o.sidx = (int64_t)(c0 + o.blk) * P.H + o.h;
  }
  return true;
}

// D = 256. Persistent CTAs, each walking blocks bid = blockIdx.x, + gridDim.x, ...
// A block is 128 rows x D of one head of one tensor. Thread 0 fetches the
// next block with one TMA copy into the other half of a shared-memory double
// buffer while the CTA works on the current one, so HBM reads stay in flight
// while the CTA rotates, reduces and stores.
//
// The work on a block: a row is spread over LPR = D/8 lanes holding 8
// consecutive elements each; the Walsh-Hadamard transform runs in registers
// (butterflies over the bits of d inside a lane, then across lanes with
// shuffles), the block amax is reduced through shared memory, and the codes
// are written with 8-byte stores.
template <int D>
__global__ void __launch_bounds__(32 * (D == 256 ? 32 : 16), D == 256 ? 1 : 2)
    fp8_prep_lanes_kernel(const __grid_constant__ PrepMaps maps, const PrepBatch pb, int total_blocks) {
  constexpr int NW = D == 256 ? 32 : 16;  // warps per CTA
  constexpr int LPR = D / 8;               // lanes per row
  constexpr int RPI = 32 / LPR;            // rows per warp instruction
  constexpr int RPW = 128 / NW;            // rows per warp
  constexpr int ITER = RPW / RPI;
  constexpr int LOG_D = D == 64 ? 6 : (D == 128 ? 7 : 8);
  constexpr uint32_t kBlockBytes = 128u * D * 2u;
  constexpr int NB = kPrepBuffers;
  extern __shared__ __align__(128) uint8_t prep_smem[];
  __shared__ float red[NW];
  __shared__ __align__(8) uint64_t full_bar[NB];
  __shared__ int gave_up;
  const uint32_t buf0 = ptx::smem_u32(prep_smem);
  const uint32_t bar0 = ptx::smem_u32(&full_bar[0]);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane / LPR;              // row of the instruction this lane serves
  const int d0 = (lane % LPR) * 8;         // first element of the lane

  if (threadIdx.x == 0) {
    for (int i = 0; i < NB; ++i) ptx::mbar_init(bar0 + 8u * i, 1);
    ptx::fence_mbar_init();
    gave_up = 0;
  }
  __syncthreads();

  // thread 0: fetch block `bid` into buffer `s` (nothing if it is skipped)
  auto fetch = [&](int bid, int s) {
    PrepBlock pbk;
    if (bid < total_blocks && prep_block(pb, bid, pbk)) {
      ptx::mbar_arrive_expect_tx(bar0 + 8u * s, kBlockBytes);
      ptx::tma_load_2d(buf0 + s * kBlockBytes, &maps.m[pbk.ti], pbk.h * D, (int)(pbk.start + pbk.blk * 128),
                       bar0 + 8u * s);
    }
  };
  // NB - 1 blocks ahead
  if (threadIdx.x == 0)
    for (int i = 0; i < NB - 1; ++i) fetch(blockIdx.x + i * gridDim.x, i);
  uint32_t phase_bits = 0u;   // bit i: parity of buffer i's next completion

  int s = 0;
  for (int bid = blockIdx.x; bid < total_blocks; bid += gridDim.x, s = (s + 1) % NB) {
    PrepBlock pbk;
    const bool live = prep_block(pb, bid, pbk);
    // block bid + (NB - 1) * gridDim.x goes into the buffer the previous
    // iteration used, free since the __syncthreads that ended it
    if (threadIdx.x == 0) fetch(bid + (NB - 1) * gridDim.x, (s + NB - 1) % NB);
    if (!live) continue;
    const PrepParams& P = pb.t[pbk.ti];
    // bounded wait for this block's copy: thread 0 waits, the CTA learns the
    // outcome at the barrier (the barrier also publishes the copied data)
    if (threadIdx.x == 0) {
      const uint64_t t0 = ptx::globaltimer_ns();
      while (!ptx::mbar_try_wait(bar0 + 8u * s, (phase_bits >> s) & 1u)) {
        if (ptx::globaltimer_ns() - t0 > 2000000000ull) {
          atomicOr(P.status, kDevTimeout | 0x40);
          gave_up = 1;
          break;
        }
      }
    }
    phase_bits ^= 1u << s;
    __syncthreads();
    if (gave_up) return;
    const uint8_t* blkmem = prep_smem + s * kBlockBytes;

    float sg[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) sg[j] = P.sigma ? (float)P.sigma[d0 + j] : 1.f;
    // 1/sqrt(D) of the rotation is applied once, in the quantisation multiplier
    const float norm = P.sigma ? rsqrtf((float)D) : 1.f;

    float x[ITER][8];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < ITER; ++i) {
      const int row = warp * RPW + i * RPI + sub;   // within the block
      if (pbk.blk * 128 + row < pbk.L) {
        cvt8(*reinterpret_cast<const uint4*>(blkmem + (row * D + d0) * 2), P.bf16, x[i]);
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
    if (threadIdx.x == 0) P.scale[pbk.sidx] = scale;

#pragma unroll
    for (int i = 0; i < ITER; ++i) {
      const int row = pbk.blk * 128 + warp * RPW + i * RPI + sub;
      if (row >= pbk.L) continue;
      *reinterpret_cast<uint2*>(P.x8 + ((pbk.start + row) * P.H + pbk.h) * D + d0) =
          make_uint2(ptx::pack_e4m3x4(x[i][0] * inv, x[i][1] * inv, x[i][2] * inv, x[i][3] * inv),
                     ptx::pack_e4m3x4(x[i][4] * inv, x[i][5] * inv, x[i][6] * inv, x[i][7] * inv));
    }
    // red[] and this buffer are reused by the next iterations
    __syncthreads();
  }
}

// ------------------------------------------------------------ D <= 128
// Two 16-bit elements -> fp32 (bf16: the bits shifted into place; fp16: the
// hardware conversion).
template <bool BF16>
__device__ __forceinline__ void cvt2(uint32_t w, float& lo, float& hi) {
  if (BF16) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xffff0000u);
  } else {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
    lo = f.x;
    hi = f.y;
  }
}

// Offset of byte `o` of a block laid out row-major in shared memory by a TMA
// copy with the 128-byte swizzle (16-byte unit bits 4..6 XOR address bits
// 7..9) or the 64-byte one (bits 4..5 XOR bits 7..8).
template <int SW>
__device__ __forceinline__ uint32_t swizzled(uint32_t o) {
  return o ^ (((o >> 7) & (SW == 128 ? 7u : 3u)) << 4);
}

// Row r of a 128 x D block (D / 64 input boxes of 64 elements x 128 rows,
// 128-byte swizzle) into v: v[i] holds elements 2i and 2i + 1. With ROT the
// row gets its sign flips (XOR of the sign bits, bit 15 of each 16-bit
// element, by mask) and the whole D-point Walsh-Hadamard transform: the
// butterfly over bit 0 of d pairs the two halves of a packed register, every
// other bit pairs two registers, so all but the first stage are f32x2 adds and
// subtracts. Returns max |x| over the row.
template <int D, bool ROT, bool BF16>
__device__ __forceinline__ float load_row(const uint8_t* blk, int r, const uint32_t* mask, uint64_t (&v)[D / 2]) {
  constexpr int NP = D / 2;
#pragma unroll
  for (int c = 0; c < D / 8; ++c) {
    const uint32_t off = (uint32_t)(c / 8) * 16384u + swizzled<128>((uint32_t)r * 128u + (uint32_t)(c % 8) * 16u);
    uint4 u = *reinterpret_cast<const uint4*>(blk + off);
    if (ROT) {
      const uint4 m = *reinterpret_cast<const uint4*>(mask + 4 * c);
      u.x ^= m.x;
      u.y ^= m.y;
      u.z ^= m.z;
      u.w ^= m.w;
    }
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float a, b;
      cvt2<BF16>(w[j], a, b);
      v[4 * c + j] = ROT ? ptx::f2pack(a + b, a - b) : ptx::f2pack(a, b);
    }
  }
  if (ROT) {
#pragma unroll
    for (int st = 1; st < NP; st <<= 1) {
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        if (i & st) continue;
        const uint64_t a = v[i], b = v[i | st];
        v[i] = ptx::add2(a, b);
        v[i | st] = ptx::sub2(a, b);
      }
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    float a, b;
    ptx::f2unpack(v[i], a, b);
    amax = ptx::max3(amax, fabsf(a), fabsf(b));
  }
  return amax;
}

// D = 64, 128. Persistent CTAs of 128 threads walk the blocks; thread r owns
// row r of the current block. Thread 0 keeps the next block's TMA copy in
// flight (two shared-memory buffers) while the CTA rotates the current one in
// registers; the block amax goes through one CTA barrier; the codes of a full
// block are written back into its buffer (its input has been read by then)
// and leave with one TMA store, those of a ragged last block with plain
// stores of the valid rows.
template <int D>
__global__ void __launch_bounds__(128, D == 64 ? 5 : 3)
    fp8_prep_rows_kernel(const __grid_constant__ PrepMaps in_maps, const __grid_constant__ PrepMaps out_maps,
                         const PrepBatch pb, int total_blocks) {
  constexpr int NP = D / 2;
  constexpr uint32_t kBlockBytes = 128u * D * 2u;
  constexpr int kOutSwizzle = D == 128 ? 128 : 64;   // the output map's swizzle (rows of D bytes)
  extern __shared__ uint8_t prep_raw[];
  __shared__ float red[4];
  __shared__ __align__(8) uint64_t full_bar[2];
  __shared__ __align__(16) uint32_t smask[3][NP];
  __shared__ int gave_up;
  // 1024-byte aligned buffers (the swizzle pattern repeats every 1024 bytes)
  const uint32_t raw = ptx::smem_u32(prep_raw);
  const uint32_t buf0 = (raw + 1023u) & ~1023u;
  uint8_t* const buf0_ptr = prep_raw + (buf0 - raw);
  const uint32_t bar0 = ptx::smem_u32(&full_bar[0]);
  const int r = threadIdx.x, warp = r >> 5, lane = r & 31;

  // sign masks of each tensor's sigma (+-1), two elements per word
  for (int i = threadIdx.x; i < 3 * NP; i += blockDim.x) {
    const int ti = i / NP, j = i % NP;
    const int8_t* sg = ti < pb.n ? pb.t[ti].sigma : nullptr;
    smask[ti][j] = sg != nullptr ? (sg[2 * j] < 0 ? 0x8000u : 0u) | (sg[2 * j + 1] < 0 ? 0x80000000u : 0u) : 0u;
  }
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar0, 1);
    ptx::mbar_init(bar0 + 8u, 1);
    ptx::fence_mbar_init();
    gave_up = 0;
  }
  __syncthreads();
  const Waiter wt{&gave_up, nullptr};

  // thread 0: fetch block `bid` into buffer `s` (nothing if it is skipped)
  auto fetch = [&](int bid, int s) -> bool {
    PrepBlock pbk;
    if (bid >= total_blocks || !prep_block(pb, bid, pbk)) return false;
    const uint32_t bar = bar0 + 8u * s;
    ptx::mbar_arrive_expect_tx(bar, kBlockBytes);
#pragma unroll
    for (int c = 0; c < D / 64; ++c)
      ptx::tma_load_2d(buf0 + s * kBlockBytes + c * 16384u, &in_maps.m[pbk.ti], pbk.h * D + c * 64,
                       (int)(pbk.start + pbk.blk * 128), bar);
    return true;
  };
  uint32_t pending = 0u;              // thread 0, bit i: a copy into buffer i is in flight
  if (threadIdx.x == 0 && fetch(blockIdx.x, 0)) pending = 1u;
  uint32_t phase_bits = 0u;           // bit i: parity of buffer i's next completion

  int s = 0;
  for (int bid = blockIdx.x; bid < total_blocks; bid += gridDim.x, s ^= 1) {
    PrepBlock pbk;
    const bool live = prep_block(pb, bid, pbk);
    if (threadIdx.x == 0) {
      // the other buffer last held the previous block's codes: its store
      // must have read them before the next block is copied in
      ptx::bulk_wait_read_all();
      if (fetch(bid + gridDim.x, s ^ 1)) pending |= 1u << (s ^ 1);
    }
    if (!live) continue;
    const PrepParams& P = pb.t[pbk.ti];
    Waiter w = wt;
    w.status = P.status;
    const bool ok = w.wait(bar0 + 8u * s, (phase_bits >> s) & 1u, 0x40);
    phase_bits ^= 1u << s;
    pending &= ~(1u << s);
    const int valid = min(128, pbk.L - pbk.blk * 128);
    uint8_t* const blk = buf0_ptr + s * kBlockBytes;

    uint64_t v[NP];
    float amax = 0.f;
    if (ok && r < valid) {
      const uint32_t* m = smask[pbk.ti];
      if (P.sigma != nullptr)
        amax = P.bf16 ? load_row<D, true, true>(blk, r, m, v) : load_row<D, true, false>(blk, r, m, v);
      else
        amax = P.bf16 ? load_row<D, false, true>(blk, r, m, v) : load_row<D, false, false>(blk, r, m, v);
    } else {
#pragma unroll
      for (int i = 0; i < NP; ++i) v[i] = 0ull;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) red[warp] = amax;
    // CTA barrier (every thread has also read its row out of the buffer) that
    // agrees on giving up if any thread's wait did
    if (__syncthreads_or(!ok)) {
      if (threadIdx.x == 0) {
        ptx::bulk_wait_all();
        for (int i = 0; i < 2; ++i)
          if ((pending >> i) & 1u) w.drain(bar0 + 8u * i, (phase_bits >> i) & 1u);
      }
      return;
    }
    // 1/sqrt(D) of the rotation is applied once, in the quantisation multiplier
    const float norm = P.sigma != nullptr ? rsqrtf((float)D) : 1.f;
    amax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3])) * norm;
    const float scale = amax > 0.f ? amax / 448.f : 1.f;
    const float inv = norm / scale;
    if (threadIdx.x == 0) P.scale[pbk.sidx] = scale;

    uint32_t code[NP / 2];
    const uint64_t inv2 = ptx::f2pack(inv, inv);
#pragma unroll
    for (int i = 0; i < NP; i += 2) {
      float a0, a1, b0, b1;
      ptx::f2unpack(ptx::mul2(v[i], inv2), a0, a1);
      ptx::f2unpack(ptx::mul2(v[i + 1], inv2), b0, b1);
      code[i / 2] = ptx::pack_e4m3x4(a0, a1, b0, b1);
    }
    const int row0 = pbk.blk * 128;
    if (valid == 128) {
#pragma unroll
      for (int c = 0; c < D / 16; ++c)
        *reinterpret_cast<uint4*>(blk + swizzled<kOutSwizzle>((uint32_t)r * D + (uint32_t)c * 16u)) =
            make_uint4(code[4 * c], code[4 * c + 1], code[4 * c + 2], code[4 * c + 3]);
      ptx::fence_proxy_async_smem();
      __syncthreads();
      if (threadIdx.x == 0) {
        ptx::tma_store_2d(&out_maps.m[pbk.ti], buf0 + s * kBlockBytes, pbk.h * D, (int)(pbk.start + row0));
        ptx::bulk_commit();
      }
    } else if (r < valid) {
      uint8_t* dst = P.x8 + ((pbk.start + row0 + r) * P.H + pbk.h) * D;
#pragma unroll
      for (int c = 0; c < D / 16; ++c)
        *reinterpret_cast<uint4*>(dst + 16 * c) =
            make_uint4(code[4 * c], code[4 * c + 1], code[4 * c + 2], code[4 * c + 3]);
    }
  }
  if (threadIdx.x == 0) ptx::bulk_wait_all();
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

cudaError_t launch_fp8_prep(const PrepParams* tensors, const CUtensorMap* in_maps, const CUtensorMap* out_maps,
                            int n_tensors, int D, int num_sms, cudaStream_t stream) {
  PrepBatch pb{};
  PrepMaps pin{}, pout{};
  long total = 0;
  pb.n = n_tensors;
  for (int i = 0; i < n_tensors; ++i) {
    pb.t[i] = tensors[i];
    pin.m[i] = in_maps[i];
    if (D <= 128) pout.m[i] = out_maps[i];
    pb.count[i] = tensors[i].B * tensors[i].H * tensors[i].nblk;
    total += pb.count[i];
  }
  if (total == 0) return cudaSuccess;
  if (total > 0x7fffffffL) return cudaErrorInvalidValue;
  cudaError_t e;
  if (D == 64 || D == 128) {
    // resident CTAs per SM: shared memory (two blocks of 128 x D 16-bit
    // elements + alignment) and registers (a row of D fp32 per thread)
    const long per_sm = D == 64 ? 5L : 3L;
    const int grid = (int)(total < per_sm * num_sms ? total : per_sm * num_sms);
    const size_t smem = 2u * 128u * (size_t)D * 2u + 1024u;
    if (D == 64) {
      e = cudaFuncSetAttribute(fp8_prep_rows_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) fp8_prep_rows_kernel<64><<<grid, 128, smem, stream>>>(pin, pout, pb, (int)total);
    } else {
      e = cudaFuncSetAttribute(fp8_prep_rows_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) fp8_prep_rows_kernel<128><<<grid, 128, smem, stream>>>(pin, pout, pb, (int)total);
    }
  } else if (D == 256) {
    // one resident CTA per SM (1024 threads, kPrepBuffers 128 x 256 blocks)
    const int grid = (int)(total < num_sms ? total : num_sms);
    const size_t smem = (size_t)kPrepBuffers * 128u * (size_t)D * 2u;
    e = cudaFuncSetAttribute(fp8_prep_lanes_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) fp8_prep_lanes_kernel<256><<<grid, 32 * 32, smem, stream>>>(pin, pb, (int)total);
  } else {
    return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace fa
