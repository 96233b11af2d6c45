// Host check of fa::tile_order: for many head counts, tiles per head and
// group sizes, every work tile index maps to a distinct (head, rank) pair in
// range, and within a group the ranks are taken in order. Prints "ok" or the
// first failing case.
#include <cstdio>
#include <vector>

#include "fa_internal.h"

int main() {
  const int bhs[] = {1, 2, 3, 5, 16, 31, 64, 100};
  const int phs[] = {1, 2, 7, 32, 65};
  const int gs[] = {1, 2, 3, 4, 8, 16};
  for (int BH : bhs)
    for (int per_head : phs)
      for (int G : gs) {
        if (G > BH) continue;
        std::vector<int> seen((size_t)BH * per_head, 0);
        int prev_group = -1, prev_rank = -1;
        for (int w = 0; w < BH * per_head; ++w) {
          int bh = -1, jj = -1;
          fa::tile_order(w, per_head, BH, G, bh, jj);
          if (bh < 0 || bh >= BH || jj < 0 || jj >= per_head || seen[(size_t)bh * per_head + jj]++) {
            std::printf("bad BH=%d per_head=%d G=%d w=%d -> (%d, %d)\n", BH, per_head, G, w, bh, jj);
            return 1;
          }
          const int group = bh / G;
          if (group == prev_group && jj < prev_rank) {
            std::printf("rank order BH=%d per_head=%d G=%d w=%d\n", BH, per_head, G, w);
            return 1;
          }
          if (group < prev_group) {
            std::printf("group order BH=%d per_head=%d G=%d w=%d\n", BH, per_head, G, w);
            return 1;
          }
          prev_group = group;
          prev_rank = jj;
        }
      }
  std::printf("ok\n");
  return 0;
}
