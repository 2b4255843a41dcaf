// Host check of the work decomposition in gqa_schedule.h (compiled with g++ by
// tests/test_schedule_cpu.py): the closed-form tile prefix and item lookup
// against brute force, and, for both schedules and many grid sizes, that every
// KV tile of every item is computed exactly once, partial slots are unique and
// owned by their CTA, and the merge side finds exactly the slots the kernel
// writes. Prints "checks=N bad=M" and exits non-zero on any mismatch.
#include "gqa_schedule.h"

#include <cstdio>
#include <map>
#include <vector>

using namespace gqa;

int main() {
  long long checks = 0;
  int bad = 0;
  const int qls[] = {1, 2, 5, 20, 21, 22, 42, 43, 127, 128, 129, 500, 512, 3072, 4096};
  const int extras[] = {0, 1, 100, 127, 128, 129, 255, 1000, 4096, 12288, 28672};
  const int grids[] = {1, 2, 3, 7, 64, 148, 152, 1000};
  for (int ql : qls)
    for (int ex : extras) {
      const Geometry geo{ql, ex, (ql + 20) / 21};
      std::vector<long long> start;
      std::vector<int> nts;
      long long acc = 0;
      for (int r = 0; r < geo.n_qtiles; ++r)
        for (int g = 0; g < 4; ++g) {
          const int nt = item_tiles(geo, geo.n_qtiles - 1 - r);
          start.push_back(acc);
          nts.push_back(nt);
          acc += nt;
        }
      const long long W = total_tiles(geo);
      if (W != acc) {
        printf("total mismatch q_len=%d p0=%d: %lld vs %lld\n", ql, ex, W, acc);
        ++bad;
      }
      for (size_t i = 0; i < start.size(); ++i)
        for (long long t = start[i]; t < start[i] + nts[i]; t += (nts[i] > 3 ? nts[i] / 3 : 1)) {
          const ItemPos p = locate(geo, t);
          ++checks;
          if (static_cast<size_t>(4 * p.r + p.g) != i || p.start != start[i] || p.nt != nts[i]) {
            if (++bad < 5) printf("locate mismatch q_len=%d p0=%d t=%lld\n", ql, ex, t);
          }
        }
      for (int mode = 0; mode < 2; ++mode)
        for (int G0 : grids) {
          const int n_items = 4 * geo.n_qtiles;
          const int G = mode == 0 ? (G0 < n_items ? G0 : n_items) : static_cast<int>(G0 < W ? G0 : W);
          std::map<long long, int> cover;  // item * 100000 + tile -> times computed
          std::map<int, int> slots;
          for (int b = 0; b < G; ++b) {
            PieceIter it;
            it.init(geo, mode, G, b, W);
            Piece w;
            while (it.next(w)) {
              const int item = 4 * (geo.n_qtiles - 1 - w.qt) + w.g;
              if (w.n0 < 0 || w.n1 > nts[item] || w.n0 >= w.n1) {
                ++bad;
                printf("bad piece range\n");
              }
              const bool whole = w.n0 == 0 && w.n1 == nts[item];
              if (whole != (w.slot < 0)) {
                ++bad;
                printf("slot / whole mismatch\n");
              }
              if (w.slot >= 0) {
                if (slots[w.slot]++) { ++bad; printf("slot reused\n"); }
                if (w.slot / 2 != b) { ++bad; printf("slot not owned by its CTA\n"); }
              }
              for (int n = w.n0; n < w.n1; ++n) cover[static_cast<long long>(item) * 100000 + n]++;
            }
          }
          for (size_t i = 0; i < nts.size(); ++i)
            for (int n = 0; n < nts[i]; ++n) {
              ++checks;
              const int c = cover[static_cast<long long>(i) * 100000 + n];
              if (c != 1 && ++bad < 10)
                printf("coverage q_len=%d p0=%d mode=%d G=%d item=%zu tile=%d count=%d\n", ql, ex,
                       mode, G, i, n, c);
            }
          if (mode == 1)
            for (int m = 1; m < G; ++m) {  // the merge kernel's view of boundary m
              const long long t = range_lo(W, G, m);
              const ItemPos p = locate(geo, t);
              if (t == p.start || range_lo(W, G, m - 1) > p.start) continue;
              const int b_lo = m - 1, b_hi = range_owner(W, G, p.start + p.nt - 1);
              if (range_lo(W, G, b_lo) > p.start || range_lo(W, G, b_hi) >= p.start + p.nt ||
                  range_lo(W, G, b_hi + 1) < p.start + p.nt) {
                ++bad;
                printf("range owner mismatch\n");
              }
              for (int b = b_lo; b <= b_hi; ++b) {
                ++checks;
                if (!slots.count(b == b_lo ? 2 * b + 1 : 2 * b)) { ++bad; printf("merge slot missing\n"); }
              }
            }
        }
    }
  printf("checks=%lld bad=%d\n", checks, bad);
  return bad != 0;
}
