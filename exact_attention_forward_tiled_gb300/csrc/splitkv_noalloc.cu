// Split-KV forward for callers that cannot allocate device memory.
//
// fa_fwd_splitkv needs a scratch buffer (the partial O and LSE of every key
// range) that its caller allocates. Some callers cannot do that: code that
// runs where cudaMalloc is not allowed or not wanted (inside a host callback,
// under an allocator that must not grow, in a plug-in that owns no memory
// pool). This entry point gives them the same computation with the scratch
// taken from a fixed array that lives in this file, so the call itself
// allocates nothing.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "fa.h"

namespace {

// The scratch: one fixed array per device that loads the library, held until
// the process exits. A problem fits when fa_fwd_splitkv_workspace_size(...)
// is at most 64 MiB: for example 31 key ranges of B=2 x H=8 x 256 query rows
// at D=128 (each range 2 MiB of fp32 partial O and 16 KiB of partial LSE).
constexpr size_t kScratchBytes = 64ull << 20;
static __device__ __align__(256) unsigned char g_splitkv_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device. In host code the array's name is only a stand-in, so the address
// must come from cudaGetSymbolAddress with that device current. The cached
// address does not survive cudaDeviceReset (the library is not to be called
// on a device after a reset).
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return FA_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_splitkv_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return FA_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FA_OK;
}

}  // namespace

extern "C" int fa_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                                      int B, int H, int Sq, int Sk, int D, float scale, int causal,
                                      int num_splits, int dtype, void* stream) {
  if (B > 0 && H > 0 && Sq > 0 && Sk >= 0) {
    const size_t need = fa_fwd_splitkv_workspace_size(B, H, Sq, Sk, D, num_splits);
    if (need > kScratchBytes) return FA_ERR_SCRATCH_LIMIT;
  }
  void* scratch = nullptr;
  const int st = scratch_address(&scratch);
  if (st != FA_OK) return st;
  // Every byte of scratch the call reads is written earlier in the same call,
  // so nothing has to be cleared between calls.
  return fa_fwd_splitkv(q, k, v, o, lse, B, H, Sq, Sk, D, scale, causal, num_splits, scratch, kScratchBytes,
                        dtype, stream);
}
