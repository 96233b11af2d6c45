// Host check of fa::SlotTable (csrc/sched_slots.h): slots are handed out in
// turn, a slot whose launch has not finished is never handed out again, a
// full table refuses, and a released or finished slot comes back. Prints
// "ok" or the first failing step.
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
  for (int i = 0; i < N; ++i) CHECK(t.take(done) == i, "fresh slots in turn");
  CHECK(t.take(done) == -1, "full table refuses");
  CHECK(t.take(done) == -1, "still full");
  finished[2] = true;
  CHECK(t.take(done) == 2, "a finished slot comes back");
  finished[2] = false;            // the new launch on slot 2 is in flight
  CHECK(t.take(done) == -1, "slot 2 held again until its new launch finishes");
  finished[0] = true;
  finished[3] = true;
  CHECK(t.take(done) == 3, "search starts after the last slot taken");
  finished[3] = false;            // its new launch is in flight
  CHECK(t.take(done) == 0, "and wraps around");
  finished[0] = false;
  CHECK(t.take(done) == -1, "full again");
  t.release(1);                   // handed out, nothing launched
  CHECK(t.take(done) == 1, "a released slot comes back");
  // many launches, each finishing before the next take: every slot is reused
  // in turn and none is ever handed out twice while held
  fa::SlotTable<N> u;
  bool live[N] = {false, false, false, false};
  auto done_u = [&](int s) { return !live[s]; };
  int last = -1;
  for (int i = 0; i < 100; ++i) {
    const int s = u.take(done_u);
    CHECK(s >= 0 && !live[s], "never a live slot");
    CHECK(s == (last + 1) % N, "round robin");
    live[s] = true;
    if (last >= 0) live[last] = false;   // the previous launch finished
    last = s;
  }
  std::printf("ok\n");
  return 0;
}
