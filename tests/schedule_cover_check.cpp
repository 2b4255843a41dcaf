// Host check of the work decomposition in gqa_schedule.h (compiled with g++ by
// tests/test_schedule_cpu.py). For many chunk shapes, grid sizes, numbers of
// whole rounds and tail splits (never more splits than the shortest item has
// KV tiles, as the planner guarantees) it checks that every KV tile of every
// item is computed exactly once, that no unit is empty, that whole items and
// only they write the output directly, that partial slots are exactly
// 0 .. tail_items*S-1 with item j's pieces in slots j*S .. j*S+S-1 (what the
// merge kernel reads), and that every unit is dealt to exactly one CTA.
// Prints "checks=N bad=M" and exits non-zero on any mismatch.
#include "gqa_schedule.h"

#include <cstdio>
#include <map>
#include <vector>

using namespace gqa;

int main() {
  long long checks = 0;
  int bad = 0;
  const int qls[] = {1, 2, 5, 20, 21, 22, 42, 43, 127, 128, 129, 500, 512, 3072, 4096};
  const int extras[] = {0, 1, 100, 127, 128, 129, 255, 1000, 4096, 28672};
  const int grids[] = {1, 2, 3, 7, 64, 152, 1000};
  const int splits[] = {1, 2, 3, 4, 7, 16};
  for (int tpi : {21, 42})
  for (int ql : qls)
    for (int ex : extras) {
      const Geometry geo{ql, ex, (ql + tpi - 1) / tpi, tpi};
      const int n_items = 4 * geo.n_qtiles;
      std::vector<int> nts;
      for (int i = 0; i < n_items; ++i) nts.push_back(item_tiles(geo, geo.n_qtiles - 1 - i / 4));
      const int shortest = item_tiles(geo, 0);
      for (int G0 : grids)
        for (int S : splits) {
          if (S > shortest) continue;
          const int max_rounds = n_items / G0;
          for (int hr : {0, 1, max_rounds}) {
            if (hr > max_rounds || (hr == 1 && max_rounds == 1 && hr != max_rounds)) continue;
            const int head = hr * G0 < n_items ? hr * G0 : n_items;
            const Schedule sc{head, S, head + (n_items - head) * S};
            const int G = G0 < sc.n_units ? G0 : sc.n_units;
            if (hr > 0 && G != G0) continue;  // whole rounds need a full grid
            std::map<long long, int> cover;
            std::map<int, int> slots;
            int units_seen = 0;
            for (int b = 0; b < G; ++b) {
              PieceIter it;
              it.init(geo, sc, G, b);
              Piece w;
              while (it.next(w)) {
                ++units_seen;
                const int item = 4 * (geo.n_qtiles - 1 - w.qt) + w.g;
                if (w.n0 < 0 || w.n1 > nts[item] || w.n0 >= w.n1) { ++bad; printf("empty or bad range\n"); }
                const bool whole = w.n0 == 0 && w.n1 == nts[item];
                if (item < head && !(whole && w.slot < 0)) { ++bad; printf("head item not whole\n"); }
                if (item >= head) {
                  if (S == 1 && w.slot >= 0) { ++bad; printf("unsplit tail wrote a slot\n"); }
                  if (S > 1) {
                    const int j = item - head;
                    if (w.slot < j * S || w.slot >= j * S + S) { ++bad; printf("slot outside item block\n"); }
                    if (slots[w.slot]++) { ++bad; printf("slot reused\n"); }
                  }
                }
                for (int n = w.n0; n < w.n1; ++n) cover[static_cast<long long>(item) * 100000 + n]++;
              }
            }
            if (units_seen != sc.n_units) { ++bad; printf("units dealt %d of %d\n", units_seen, sc.n_units); }
            for (int i = 0; i < n_items; ++i)
              for (int n = 0; n < nts[i]; ++n) {
                ++checks;
                const int c = cover[static_cast<long long>(i) * 100000 + n];
                if (c != 1 && ++bad < 10)
                  printf("coverage q_len=%d p0=%d G=%d S=%d hr=%d item=%d tile=%d count=%d\n", ql, ex,
                         G, S, hr, i, n, c);
              }
            if (S > 1 && static_cast<int>(slots.size()) != (n_items - head) * S) {
              ++bad;
              printf("slot count\n");
            }
          }
        }
    }
  printf("checks=%lld bad=%d\n", checks, bad);
  return bad != 0;
}
