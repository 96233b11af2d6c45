// Host check of fa::SlotTable (csrc/sched_slots.h): slots are handed out in
// turn, a slot whose launch has not finished is never handed out as free,
// a full table hands out the slot handed out longest ago with wait = true,
// and a released or finished slot comes back. Prints "ok" or the first
// failing step.
#include <cstdio>

#include "sched_slots.h"

#define CHECK(cond, what)                 \
  do {                                    \
    if (!(cond)) {                        \
      std::printf("fail: %s\n", what);    \
      return 1;                           \
    }                                     \
  } while (0)

int main() {
  constexpr int N = 4;
  fa::SlotTable<N> t;
  bool finished[N] = {false, false, false, false};
  auto done = [&](int s) { return finished[s]; };
  bool wait = true;
  for (int i = 0; i < N; ++i) {
    CHECK(t.take(done, wait) == i && !wait, "fresh slots in turn, no wait");
  }
  CHECK(t.take(done, wait) == 0 && wait, "full table: the oldest slot, with a wait");
  CHECK(t.take(done, wait) == 1 && wait, "still full: the next oldest, with a wait");
  finished[3] = true;
  CHECK(t.take(done, wait) == 3 && !wait, "a finished slot comes back without a wait");
  finished[3] = false;            // the new launch on slot 3 is in flight
  CHECK(t.take(done, wait) == 0 && wait, "all held again: wraps to the oldest");
  finished[2] = true;
  CHECK(t.take(done, wait) == 2 && !wait, "a finished slot is preferred to a wait");
  finished[2] = false;
  t.release(3);                   // handed out free, nothing launched
  CHECK(t.take(done, wait) == 3 && !wait, "a released slot comes back");
  // an untracked (captured) launch neither queries nor marks anything
  fa::SlotTable<N> c;
  int queries = 0;
  auto count = [&](int) { ++queries; return false; };
  CHECK(c.untracked() == 0 && c.untracked() == 1, "untracked slots in turn");
  CHECK(c.take(count, wait) == 2 && !wait && queries == 0, "untracked slots stay free");
  // a deep single-stream queue: every take after the first N waits for the
  // slot handed out N launches earlier, so no two launches that may overlap
  // share a slot
  fa::SlotTable<N> u;
  int holder[N] = {-1, -1, -1, -1};   // launch index that last took the slot
  auto never = [&](int) { return false; };
  for (int i = 0; i < 100; ++i) {
    const int s = u.take(never, wait);
    CHECK(s == i % N, "round robin");
    CHECK(wait == (i >= N), "a wait exactly when the slot is held");
    CHECK(!wait || holder[s] == i - N, "the wait is for the launch N earlier");
    holder[s] = i;
  }
  std::printf("ok\n");
  return 0;
}
