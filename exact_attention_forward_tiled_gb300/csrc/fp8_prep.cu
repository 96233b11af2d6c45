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
// with reads in flight throughout. A thread owns a whole row (D <= 128) or
// half of one (D = 256) and runs the Walsh-Hadamard transform on packed fp32
// pairs in its registers; at D = 256 the last butterfly crosses to the
// neighbouring lane.
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

struct PrepMaps {
  CUtensorMap m[3];
};

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

// E elements of row r of a 128 x D block (D / 64 input boxes of 64 elements
// x 128 rows, 128-byte swizzle), starting at element e0 (0, or 128 for the
// second half of a D = 256 row), into v: v[i] holds elements e0 + 2i and
// e0 + 2i + 1. With ROT the elements get their sign flips (XOR of the sign
// bits, bit 15 of each 16-bit element, by mask) and the E-point
// Walsh-Hadamard transform: the butterfly over bit 0 of d pairs the two
// halves of a packed register, every other bit pairs two registers, so all but
// the first stage are f32x2 adds and subtracts. Returns max |x| over the E
// elements (before any stage that crosses to another thread).
template <int E, bool ROT, bool BF16>
__device__ __forceinline__ float load_row(const uint8_t* blk, int r, int e0, const uint32_t* mask,
                                          uint64_t (&v)[E / 2]) {
  constexpr int NP = E / 2;
#pragma unroll
  for (int c = 0; c < E / 8; ++c) {
    const int e = e0 + 8 * c;
    const uint32_t off =
        (uint32_t)(e / 64) * 16384u + swizzled<128>((uint32_t)r * 128u + (uint32_t)((e % 64) / 8) * 16u);
    uint4 u = *reinterpret_cast<const uint4*>(blk + off);
    if (ROT) {
      const uint4 m = *reinterpret_cast<const uint4*>(mask + e / 2);
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

// Persistent CTAs walk the blocks; each row of the current block belongs to
// TPR threads (1, or 2 at D = 256), each of which owns E = D / TPR elements of
// it. Thread 0 keeps the next block's TMA copy in flight (two shared-memory
// buffers) while the CTA rotates the current one in registers; the block amax
// goes through one CTA barrier; the codes of a full block are written back
// into its buffer (its input has been read by then) and leave with TMA stores,
// those of a ragged last block with plain stores of the valid rows.
template <int D>
struct PrepCfg {
  static constexpr int TPR = D == 256 ? 2 : 1;           // threads per row
  static constexpr int E = D / TPR;                        // elements per thread
  static constexpr int kThreads = 128 * TPR;
  static constexpr int kCtasPerSm = D == 64 ? 5 : (D == 128 ? 3 : 1);
  static constexpr uint32_t kBlockBytes = 128u * D * 2u;   // one 16-bit input block
  static constexpr int kOutBox = D == 64 ? 64 : 128;       // bytes per row of an output box
  static constexpr int kOutSwizzle = kOutBox;              // that box's swizzle (64 or 128 bytes)
  static constexpr size_t kSmemBytes = 2u * kBlockBytes + 1024u;
};

template <int D>
__global__ void __launch_bounds__(PrepCfg<D>::kThreads, PrepCfg<D>::kCtasPerSm)
    fp8_prep_kernel(const __grid_constant__ PrepMaps in_maps, const __grid_constant__ PrepMaps out_maps,
                    const PrepBatch pb, int total_blocks) {
  using C = PrepCfg<D>;
  constexpr int E = C::E, NP = E / 2, NW = C::kThreads / 32;
  constexpr uint32_t kBlockBytes = C::kBlockBytes;
  extern __shared__ uint8_t prep_raw[];
  __shared__ float red[NW];
  __shared__ __align__(8) uint64_t full_bar[2];
  __shared__ __align__(16) uint32_t smask[3][D / 2];
  __shared__ int gave_up;
  // 1024-byte aligned buffers (the swizzle pattern repeats every 1024 bytes)
  const uint32_t raw = ptx::smem_u32(prep_raw);
  const uint32_t buf0 = (raw + 1023u) & ~1023u;
  uint8_t* const buf0_ptr = prep_raw + (buf0 - raw);
  const uint32_t bar0 = ptx::smem_u32(&full_bar[0]);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = threadIdx.x / C::TPR;        // row of the block
  const int half = threadIdx.x % C::TPR;     // which E elements of it (partner: the next lane)
  const int e0 = half * E;

  // sign masks of each tensor's sigma (+-1), two elements per word
  for (int i = threadIdx.x; i < 3 * (D / 2); i += blockDim.x) {
    const int ti = i / (D / 2), j = i % (D / 2);
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
      // the other buffer last held the previous block's codes: its stores
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
    const bool rot = P.sigma != nullptr;

    uint64_t v[NP];
    float amax = 0.f;
    if (ok && r < valid) {
      const uint32_t* m = smask[pbk.ti];
      if (rot)
        amax = P.bf16 ? load_row<E, true, true>(blk, r, e0, m, v) : load_row<E, true, false>(blk, r, e0, m, v);
      else
        amax = P.bf16 ? load_row<E, false, true>(blk, r, e0, m, v) : load_row<E, false, false>(blk, r, e0, m, v);
    } else {
#pragma unroll
      for (int i = 0; i < NP; ++i) v[i] = 0ull;
    }
    if (C::TPR == 2 && rot) {
      // butterfly over bit 7 of d: the lower half becomes mine + other, the
      // upper half other - mine (one FMA each with the sign of the half);
      // both lanes of a row take the same branch (rot is per block)
      const uint64_t sgn = half ? ptx::f2pack(-1.f, -1.f) : ptx::f2pack(1.f, 1.f);
      amax = 0.f;
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        const uint64_t other = __shfl_xor_sync(0xffffffffu, v[i], 1);
        v[i] = ptx::fma2(v[i], sgn, other);
        float a, b;
        ptx::f2unpack(v[i], a, b);
        amax = ptx::max3(amax, fabsf(a), fabsf(b));
      }
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
    // 1/sqrt(D) of the rotation, rounded once to fp32 (exact for D = 64 and
    // 256), is applied once, in the quantisation multiplier; every step of the
    // code decision is then a correctly rounded fp32 operation
    const float norm = rot ? (D == 64 ? 0.125f : D == 128 ? 0x1.6a09e6p-4f : 0.0625f) : 1.f;
    amax = red[0];
#pragma unroll
    for (int i = 1; i < NW; ++i) amax = fmaxf(amax, red[i]);
    amax *= norm;
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
      // codes in the output boxes' layout (D / kOutBox boxes of kOutBox-byte
      // rows, each box 128 rows), then one TMA store per box
#pragma unroll
      for (int c = 0; c < E / 16; ++c) {
        const int e = e0 + 16 * c;
        const uint32_t off = (uint32_t)(e / C::kOutBox) * (128u * C::kOutBox) +
                             swizzled<C::kOutSwizzle>((uint32_t)r * C::kOutBox + (uint32_t)(e % C::kOutBox));
        *reinterpret_cast<uint4*>(blk + off) = make_uint4(code[4 * c], code[4 * c + 1], code[4 * c + 2], code[4 * c + 3]);
      }
      ptx::fence_proxy_async_smem();
      __syncthreads();
      if (threadIdx.x == 0) {
#pragma unroll
        for (int b = 0; b < D / C::kOutBox; ++b)
          ptx::tma_store_2d(&out_maps.m[pbk.ti], buf0 + s * kBlockBytes + b * (128u * C::kOutBox),
                            pbk.h * D + b * C::kOutBox, (int)(pbk.start + row0));
        ptx::bulk_commit();
      }
    } else if (r < valid) {
      uint8_t* dst = P.x8 + ((pbk.start + row0 + r) * P.H + pbk.h) * D + e0;
#pragma unroll
      for (int c = 0; c < E / 16; ++c)
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
    pout.m[i] = out_maps[i];
    pb.count[i] = tensors[i].B * tensors[i].H * tensors[i].nblk;
    total += pb.count[i];
  }
  if (total == 0) return cudaSuccess;
  if (total > 0x7fffffffL) return cudaErrorInvalidValue;
  // resident CTAs per SM: shared memory (two 128 x D blocks of 16-bit
  // elements + alignment) and registers (E fp32 per thread)
  auto run = [&](auto kern, int threads, int per_sm, size_t smem) -> cudaError_t {
    const int grid = (int)(total < (long)per_sm * num_sms ? total : (long)per_sm * num_sms);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) kern<<<grid, threads, smem, stream>>>(pin, pout, pb, (int)total);
    return e;
  };
  cudaError_t e;
  switch (D) {
    case 64:
      e = run(fp8_prep_kernel<64>, PrepCfg<64>::kThreads, PrepCfg<64>::kCtasPerSm, PrepCfg<64>::kSmemBytes);
      break;
    case 128:
      e = run(fp8_prep_kernel<128>, PrepCfg<128>::kThreads, PrepCfg<128>::kCtasPerSm, PrepCfg<128>::kSmemBytes);
      break;
    case 256:
      e = run(fp8_prep_kernel<256>, PrepCfg<256>::kThreads, PrepCfg<256>::kCtasPerSm, PrepCfg<256>::kSmemBytes);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace fa
