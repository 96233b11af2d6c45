// Internal interface between the C-ABI front end (fa_api.cu) and the kernel
// translation units (one per head dimension, compiled in parallel).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Device status word values (bit-or'ed with the role that gave up).
enum : int {
  kDevOk = 0,
  kDevTimeout = 0x100,     // an mbarrier wait exceeded its time limit (low bits: where)
  kDevBadSeqlens = 0x200,  // a varlen sequence broke its declared bounds (skipped)
};

// Everything the forward kernel needs besides the three tensor maps.
struct FwdParams {
  void* o;                 // [tokens_q, H, D] output, same 16-bit type as Q
  float* lse;              // fixed: [B, H, Sq]; varlen: [H, total_q]
  const int* cu_q;         // varlen prefix sums [B + 1] (device) or nullptr
  const int* cu_k;
  int B, H, Sq, Sk;        // fixed lengths, or (varlen) max lengths
  int total_q, total_k;    // rows of the Q/O and K/V tensors
  int n_qblk;              // CTA query blocks per (sequence, head)
  int ntiles;              // B * H * n_qblk
  float c;                 // softmax scale * log2(e)
  int* status;             // device status word
  // dynamic tile scheduler: {next tile, CTAs done}; zero at launch, and the
  // last CTA to finish puts both back to zero
  unsigned int* sched;
  // e4m3 inputs only: fp32 block scales [B, H, nblk] of Q', K', V (one per
  // 128-row block of a head); real value = code value * scale
  const float* q_scale;
  const float* k_scale;
  const float* v_scale;
  int nblk_q, nblk_k;
  // split-KV: the keys of every (sequence, head) are cut into n_split ranges
  // of split_blocks 128-key blocks; each work tile covers one range and writes
  // a partial, self-normalised fp32 O and its LSE into o_part / lse_part
  // ([n_split, tokens_q, H, D] and [n_split, B, H, Sq]). n_split = 1 and
  // o_part = nullptr: no split, O and LSE are written directly.
  int n_split, split_blocks;
  float* o_part;
  float* lse_part;
  // e4m3 varlen: prefix sums of the per-sequence 128-row block counts; the
  // scales are then [cu_blocks[B], H] (nullptr: fixed length, [B, H, nblk])
  const int* cu_blocks_q;
  const int* cu_blocks_k;
  // paged K/V (block_table == nullptr: contiguous). The K and V tensor maps
  // cover the caches as [num_pages * page_size, H * D] rows; key j of
  // sequence b is row block_table[b * max_pages + j / page_size] * page_size
  // + j % page_size. seqlens_k [B]: keys of each sequence. page_rows =
  // min(page_size, 128) rows per TMA box.
  const int* block_table;
  const int* seqlens_k;
  int max_pages, page_size, num_pages, page_rows;
  int page_shift;   // log2(page_size) for a power of two, else -1
  int n_kblk_tag;   // max_pages * page_size / 128 + 1: tags a (sequence, key block) pair
  int head_group;   // heads whose tiles are visited rank-major together (tile_order)
#ifdef FA_TEST_WITHHOLD_KV
  int test_withhold_kb;   // test build only: key block whose K tile CTA 0 never loads (-1: none)
#endif
};

// Work tile w -> (sequence-head index bh, rank jj of the tile within its
// head) for B*H heads of per_head tiles each. Heads go in groups of G; within
// a group the tiles are taken rank by rank (rank 0 of every head of the group,
// then rank 1, ...), so with ranks ordered from the most expensive tile down
// (causal) the last tiles handed out are the cheapest ones and the run ends
// without a long tile running alone, while the heads in flight at one time
// (about one group) keep their streamed K/V in L2. G = 1: head by head.
// A bijection of [0, BH * per_head) for every G >= 1.
__host__ __device__ inline void tile_order(int w, int per_head, int BH, int G, int& bh, int& jj) {
  if (G <= 1) {
    bh = w / per_head;
    jj = w - bh * per_head;
    return;
  }
  const int g0 = (w / (G * per_head)) * G;        // first head of w's group
  const int gn = BH - g0 < G ? BH - g0 : G;        // heads in that group
  const int r = w - g0 * per_head;
  jj = r / gn;
  bh = g0 + (r - jj * gn);
}

// Element kinds of the attention inputs.
enum Kind : int { kF16 = 0, kBF16 = 1, kE4M3 = 2 };

// Per-launch description filled by the front end.
struct FwdLaunch {
  CUtensorMap tq, tk, tv;
  CUtensorMap to;   // O [tokens, H * D], 16-bit, boxes of 64 x 128 with the 128-byte swizzle (TMA stores)
  FwdParams p;
  int D;
  int kind;  // Kind
  bool causal;
  bool one_tile;  // D <= 128 with one query tile per work tile (short queries)
  int num_sms;
  cudaStream_t stream;
};

// Rows of Q per CTA for head dimension D (2 x 128 for D <= 128, 128 for 256).
constexpr int cta_rows(int D) { return D <= 128 ? 256 : 128; }
// 16-bit inputs: query sequences of at most 128 rows (decode, short chunks)
// take the one-query-tile configuration at every D, so no work tile carries
// a second, empty query tile through the MMAs and the softmax.
constexpr int cta_rows16(int D, int Sq) { return (D <= 128 && Sq > 128) ? 256 : 128; }

cudaError_t launch_fwd_d64(const FwdLaunch& L);
cudaError_t launch_fwd_d128(const FwdLaunch& L);
cudaError_t launch_fwd_d64_q1(const FwdLaunch& L);
cudaError_t launch_fwd_d128_q1(const FwdLaunch& L);
cudaError_t launch_fwd_d256(const FwdLaunch& L);
cudaError_t launch_splitkv_merge(const float* o_part, const float* lse_part, void* o, float* lse,
                                 int n_split, int B, int H, int Sq, int D, int out_fp16, int num_sms,
                                 cudaStream_t stream);
cudaError_t launch_fwd_fp8_d64(const FwdLaunch& L);
cudaError_t launch_fwd_fp8_d128(const FwdLaunch& L);
cudaError_t launch_fwd_fp8_d256(const FwdLaunch& L);

// Backward pass. Both kernels are one template in two orientations: a
// 128-row block of the "resident" side (R1, R2) stays in shared memory while
// 128-row blocks of the "streamed" side (T1, T2) pass through.
//   dQ kernel:   R1 = Q, R2 = dO, T1 = K, T2 = V   -> dr1 = dQ
//   dK/dV kernel: R1 = K, R2 = V, T1 = Q, T2 = dO  -> dr1 = dK, dr2 = dV
struct BwdParams {
  void* dr1;               // [tokens_R, H, D] gradient of the resident side, input type
  void* dr2;               // dV (dK/dV kernel), else nullptr
  const float* lse2;       // [H, total_q]: LSE * log2(e), +inf for rows with no key
  const float* delta;      // [H, total_q]: rowsum(dO * O)
  const int* cu_q;         // varlen prefix sums [B + 1] (device) or nullptr
  const int* cu_k;
  int B, H, Sq, Sk;        // fixed lengths, or (varlen) max lengths
  int total_q, total_k;
  int n_rblk;              // resident 128-row blocks per (sequence, head)
  int ntiles;              // B * H * n_rblk
  float c;                 // softmax scale * log2(e)
  float scale;             // softmax scale (the factor of dQ and dK)
  int* status;
  unsigned int* sched;
  int head_group;          // heads whose tiles are visited rank-major together (tile_order)
};

struct BwdLaunch {
  CUtensorMap tr1, tr2, tt1, tt2;
  BwdParams p;
  int D;
  int kind;  // kF16 or kBF16
  bool causal;
  bool dq;   // true: dQ kernel, false: dK/dV kernel
  int part;  // D = 256 dK/dV side, one kernel each: 1 dK, 2 dV (0 below D = 256: both)
  int num_sms;
  cudaStream_t stream;
};

cudaError_t launch_bwd_d64(const BwdLaunch& L);
cudaError_t launch_bwd_d128(const BwdLaunch& L);
cudaError_t launch_bwd_d256(const BwdLaunch& L);
// lse2 / delta of every (query token, head) from O, dO and the forward's LSE
// (lse_varlen: LSE is [H, total_q], else [B, H, Sq])
cudaError_t launch_bwd_prep(const void* o, const void* dout, const float* lse, float* lse2, float* delta,
                            int total_q, int H, int D, int Sq, int lse_varlen, int fp16, cudaStream_t stream);

// FP8 preparation: rotation (optional) + block quantisation of one tensor.
struct PrepParams {
  const void* x;        // [tokens, H, D] 16-bit input
  uint8_t* x8;          // [tokens, H, D] e4m3 output
  float* scale;         // fixed: [B, H, nblk]; varlen: [cu_blocks[B], H] fp32 output
  const int8_t* sigma;  // [D] +-1, or nullptr: no rotation
  int B, H, S, nblk;    // varlen: S = max length, nblk = ceil(S / 128)
  int bf16;             // 1: bf16 input, 0: fp16
  const int* cu_seqlens;  // varlen: [B + 1] token prefix sums, or nullptr
  const int* cu_blocks;   // varlen: [B + 1] prefix sums of ceil(L_b / 128)
  int total;              // varlen: rows of x
  int* status;            // device status word (bad cu_seqlens entries)
};
cudaError_t launch_varlen_blocks(const int* cu_seqlens, int B, int* cu_blocks, cudaStream_t stream);
// in_maps: [rows, H * D] tensor maps of the 16-bit inputs, boxes of 64
// elements x 128 rows with the 128-byte swizzle. out_maps: [rows, H * D] maps
// of the e4m3 outputs, boxes of min(D, 128) bytes x 128 rows, 64-byte swizzle
// for D = 64, 128-byte otherwise.
cudaError_t launch_fp8_prep(const PrepParams* tensors, const CUtensorMap* in_maps, const CUtensorMap* out_maps,
                            int n_tensors, int D, int num_sms, cudaStream_t stream);

}  // namespace fa
