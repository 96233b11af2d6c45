// Synchronisation pieces shared by the attention kernels: bounded mbarrier
// waits (every wait gives up after kWaitLimitNs, records where in the device
// status word and raises a CTA-wide abort flag) and the shared-memory ring
// through which a load warp hands work-tile indices to the other roles.
#pragma once

#include <cstdint>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

#ifdef FA_TEST_WITHHOLD_KV
// test build (see load_role): waits give up after 50 ms, so the test that
// withholds a tile sees the timeout quickly
constexpr uint64_t kWaitLimitNs = 50000000ull;
#else
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait
#endif
constexpr float kLn2 = 0.6931471805599453f;

// Bounded mbarrier waits shared by all roles of a CTA.
struct Waiter {
  volatile int* abort_flag;
  int* status;

  __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, int where) const {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t n = 1;; ++n) {
      if (ptx::mbar_try_wait(bar, parity)) return true;
      if ((n & 63u) == 0) {
        if (*abort_flag) return false;
        if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
          *abort_flag = 1;
          atomicOr(status, kDevTimeout | where);
          return false;
        }
      }
    }
  }
  // Whole-warp wait: every lane waits; the warp proceeds only if all did.
  __device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, int where) const {
    const bool ok = wait(bar, parity, where);
    return __all_sync(0xffffffffu, ok);
  }
  // Drain wait used on the way out: bounded, ignores the abort flag.
  __device__ __forceinline__ void drain(uint32_t bar, uint32_t parity) const {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
      if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) return;
    }
  }
};

// Work-tile hand-off. The load warp fetches tile indices -- the first one is
// blockIdx.x, later ones come from a global atomic counter so CTAs that drew
// light tiles (causal, varlen) take more -- and publishes them in a small
// shared-memory ring; the MMA thread and every softmax warp read the same
// sequence from it. -1 ends the sequence.
struct TileRing {
  uint32_t full0, empty0;   // barrier addresses of slot 0
  volatile int* slots;

  __device__ __forceinline__ uint32_t full(int s) const { return full0 + 8u * s; }
  __device__ __forceinline__ uint32_t empty(int s) const { return empty0 + 8u * s; }
};

// Next tile from the ring for a consumer; false at the end of the sequence
// or when the CTA gives up. `lead` lanes arrive on the slot's empty barrier.
__device__ __forceinline__ bool next_tile(const TileRing& ring, const Waiter& wt, int j, int ring_len,
                                          bool warp_wide, bool lead, int& w) {
  const int rs = j % ring_len;
  const uint32_t par = (j / ring_len) & 1u;
  const bool ok = warp_wide ? wt.wait_warp(ring.full(rs), par, 10) : wt.wait(ring.full(rs), par, 10);
  if (!ok) return false;
  w = ring.slots[rs];
  if (warp_wide) __syncwarp();
  if (lead) ptx::mbar_arrive(ring.empty(rs));
  return w >= 0;
}

}  // namespace fa
