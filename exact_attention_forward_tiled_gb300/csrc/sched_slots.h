// Launch slots of the tile scheduler. Every persistent launch needs its own
// pair of device counters {next tile, CTAs done} that start at zero; the
// library keeps a fixed set of pairs per device (static __device__ arrays)
// and the last CTA of a launch puts its pair back to zero. Two launches that
// run at the same time must never share a pair, or they would skip or repeat
// tiles.
//
// SlotTable hands out slots in turn, skipping any still held by a launch in
// flight. When every slot is held it hands out the slot at `next` anyway --
// the one handed out longest ago -- and says so (`wait` = true): the caller
// must then order its launch after that slot's previous launch (an event
// wait on its stream, done on the GPU), so that the two never run at once.
// Whether a launch has finished is the caller's question to answer (a CUDA
// event query on the device, a flag in the host test); plain host code, no
// CUDA types.
#pragma once

namespace fa {

template <int N>
struct SlotTable {
  bool held[N] = {};   // the slot was handed out and its launch may still run
  int next = 0;        // where the search for a free slot starts

  // The first slot from `next` on that is free: never handed out, or its
  // launch finished (done(s) is true); wait = false. When all N are still
  // held: the slot at `next`, still held by its previous launch, and
  // wait = true.
  template <class Done>
  int take(Done&& done, bool& wait) {
    for (int k = 0; k < N; ++k) {
      const int s = (next + k) % N;
      if (!held[s] || done(s)) {
        held[s] = true;
        next = (s + 1) % N;
        wait = false;
        return s;
      }
    }
    const int s = next;
    next = (s + 1) % N;
    wait = true;
    return s;
  }

  // A slot for a launch that is not tracked (one captured into a graph):
  // the slot at `next`, with no query and no change to what is held.
  int untracked() {
    const int s = next;
    next = (s + 1) % N;
    return s;
  }

  // A slot handed out free (wait = false) had nothing launched with it.
  void release(int s) {
    if (s >= 0 && s < N) held[s] = false;
  }
};

}  // namespace fa
