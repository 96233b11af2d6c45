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
  uint32_t* tile_counter;  // unused by the static scheduler (reserved)
};

// Per-launch description filled by the front end.
struct FwdLaunch {
  CUtensorMap tq, tk, tv;
  FwdParams p;
  int D;
  bool fp16;
  bool causal;
  int num_sms;
  cudaStream_t stream;
};

// Rows of Q per CTA for head dimension D (2 x 128 for D <= 128, 128 for 256).
constexpr int cta_rows(int D) { return D <= 128 ? 256 : 128; }

cudaError_t launch_fwd_d64(const FwdLaunch& L);
cudaError_t launch_fwd_d128(const FwdLaunch& L);
cudaError_t launch_fwd_d256(const FwdLaunch& L);

}  // namespace fa
