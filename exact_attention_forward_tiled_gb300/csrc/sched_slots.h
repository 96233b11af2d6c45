// Launch slots of the tile scheduler. Every persistent launch needs its own
// pair of device counters {next tile, CTAs done} that start at zero; the
// library keeps a fixed set of pairs per device (static __device__ arrays)
// and the last CTA of a launch puts its pair back to zero. A slot may be
// handed to a new launch only once the launch that last held it has
// finished, or two launches would share counters and skip or repeat tiles.
//
// SlotTable hands out slots in turn, skipping any still held, and returns
// -1 when every slot is held by a launch in flight: the caller then refuses
// the launch instead of reusing a live pair. Whether a launch has finished
// is the caller's question to answer (a CUDA event query on the device, a
// flag in the host test); plain host code, no CUDA types.
#pragma once

namespace fa {

template <int N>
struct SlotTable {
  bool held[N] = {};   // the slot was handed out and its launch may still run
  int next = 0;        // where the search for a free slot starts

  // The first slot from `next` on that is free: never handed out, or its
  // launch finished (done(s) is true). -1 when all N are still held.
  template <class Done>
  int take(Done&& done) {
    for (int k = 0; k < N; ++k) {
      const int s = (next + k) % N;
      if (!held[s] || done(s)) {
        held[s] = true;
        next = (s + 1) % N;
        return s;
      }
    }
    return -1;
  }

  // The slot was handed out but nothing was launched with it.
  void release(int s) {
    if (s >= 0 && s < N) held[s] = false;
  }
};

}  // namespace fa
