// Host check of the work decomposition in gqa_schedule.h (compiled with g++ by
// tests/test_schedule_cpu.py). For many chunk shapes and seeded batches of
// several sequences (item numbering inverted by item_of), grid sizes, numbers of
// whole rounds and tail splits (never more splits than the shortest item has
// KV tiles, as the planner guarantees) it checks that every KV tile of every
// item is computed exactly once, that no unit is empty, that whole items and
// only they write the output directly, that partial slots are exactly
// 0 .. tail_items*S-1 with item j's pieces in slots j*S .. j*S+S-1 (what the
// merge kernel reads), and that every unit is dealt to exactly one CTA.
// The balanced tail (S = 0) is checked the same way, and against the merge
// kernel's view of it: for every tail item, balanced_item_pieces /
// balanced_slot must name exactly the workers and slots that wrote its pieces,
// in KV order, and an item they call unsplit must have been written whole.
// Prints "checks=N bad=M" and exits non-zero on any mismatch.
#include "gqa_schedule.h"

#include <cstdint>
#include <cstdio>
#include <map>
#include <utility>
#include <vector>

using namespace gqa;

namespace {

long long checks = 0;
int bad = 0;

uint32_t lcg(uint32_t& s) {
  s = s * 1664525u + 1013904223u;
  return s >> 8;
}

// A call's sequence table (any order: coverage must not depend on it).
void make_batch(const std::vector<std::pair<int, int>>& lens, int tpi, Batch& b) {
  b.n_seq = 0;
  b.tok_per_item = tpi;
  int items = 0, q_start = 0, kv_start = 0;
  for (size_t i = 0; i < lens.size(); ++i) {
    const int ql = lens[i].first, kl = lens[i].second;
    if (ql > 0) {
      const int nq = (ql + tpi - 1) / tpi;
      b.seq[b.n_seq++] = SeqGeo{q_start, ql, kv_start, kl, nq, items, static_cast<int>(i), 0};
      items += 4 * nq;
    }
    q_start += ql;
    kv_start += kl;
  }
  b.n_items = items;
}

void check_balanced(const Batch& b, const std::vector<int>& nts, const std::vector<long long>& off,
                    const int* grids, int n_grids);

void check_batch(const Batch& b, const int* grids, int n_grids, const int* splits, int n_splits) {
  const int n_items = b.n_items;
  std::vector<int> nts(static_cast<size_t>(n_items));
  int shortest = 1 << 30;
  std::vector<long long> off(static_cast<size_t>(n_items) + 1, 0);  // first tile of each item
  for (int i = 0; i < n_items; ++i) {  // item_of must invert item numbering
    int seq, qt, g;
    item_of(b, i, seq, qt, g);
    const SeqGeo& s = b.seq[seq];
    const int li = 4 * (s.n_qtiles - 1 - qt) + g;
    if (s.item_begin + li != i || qt < 0 || qt >= s.n_qtiles) { ++bad; printf("item_of\n"); }
    nts[static_cast<size_t>(i)] = item_tiles(s, b.tok_per_item, qt);
    off[static_cast<size_t>(i) + 1] = off[static_cast<size_t>(i)] + nts[static_cast<size_t>(i)];
    if (nts[static_cast<size_t>(i)] < shortest) shortest = nts[static_cast<size_t>(i)];
  }
  for (int gi = 0; gi < n_grids; ++gi)
    for (int si = 0; si < n_splits; ++si) {
      const int G0 = grids[gi], S = splits[si];
      if (S > shortest) continue;
      const int max_rounds = n_items / G0;
      for (int hr : {0, 1, max_rounds}) {
        if (hr > max_rounds) continue;
        const int head = hr * G0 < n_items ? hr * G0 : n_items;
        const Schedule sc{head, S, head + (n_items - head) * S, 0};
        const int G = G0 < sc.n_units ? G0 : sc.n_units;
        if (hr > 0 && G != G0) continue;  // whole rounds need a full grid
        std::vector<int> cover(static_cast<size_t>(off[static_cast<size_t>(n_items)]), 0);
        std::map<int, int> slots;
        int units_seen = 0;
        for (int x = 0; x < G; ++x) {
          PieceIter it;
          it.init(&b, nullptr, sc, G, x);
          Piece w;
          while (it.next(w)) {
            ++units_seen;
            const SeqGeo& s = b.seq[w.seq];
            const int item = s.item_begin + 4 * (s.n_qtiles - 1 - w.qt) + w.g;
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
            for (int n = w.n0; n < w.n1; ++n) cover[static_cast<size_t>(off[static_cast<size_t>(item)] + n)]++;
          }
        }
        if (units_seen != sc.n_units) { ++bad; printf("units dealt %d of %d\n", units_seen, sc.n_units); }
        for (int i = 0; i < n_items; ++i)
          for (int n = 0; n < nts[static_cast<size_t>(i)]; ++n) {
            ++checks;
            const int c = cover[static_cast<size_t>(off[static_cast<size_t>(i)] + n)];
            if (c != 1 && ++bad < 10)
              printf("coverage seqs=%d G=%d S=%d hr=%d item=%d tile=%d count=%d\n", b.n_seq, G, S,
                     hr, i, n, c);
          }
        if (S > 1 && static_cast<int>(slots.size()) != (n_items - head) * S) {
          ++bad;
          printf("slot count\n");
        }
      }
    }
  check_balanced(b, nts, off, grids, n_grids);
}

struct Emitted {
  int x, n0, n1, slot;
};

void check_balanced(const Batch& b, const std::vector<int>& nts, const std::vector<long long>& off,
                    const int* grids, int n_grids) {
  static TailPrefix tp;
  const int n_items = b.n_items;
  for (int gi = 0; gi < n_grids; ++gi) {
    const int max_rounds = n_items / grids[gi];
    for (int hr : {0, 1, max_rounds}) {
      if (hr > max_rounds) continue;
      int G = grids[gi];
      const int head = hr * G < n_items ? hr * G : n_items;
      const int n_tail = n_items - head;
      if (n_tail < 1 || n_tail > kMaxBalancedTail) continue;
      tp.v[0] = 0;
      for (int k = 0; k < n_tail; ++k) tp.v[k + 1] = tp.v[k] + nts[static_cast<size_t>(head + k)];
      const long long W = tp.v[n_tail];
      if (hr == 0 && W < G) G = static_cast<int>(W);  // the planner shrinks the grid
      if (W < G) continue;
      const Schedule sc{head, 0, 0, n_tail};
      std::vector<int> cover(static_cast<size_t>(off[static_cast<size_t>(n_items)]), 0);
      std::map<int, int> slots;
      std::vector<std::vector<Emitted>> by_item(static_cast<size_t>(n_tail));
      for (int x = 0; x < G; ++x) {
        PieceIter it;
        it.init(&b, tp.v, sc, G, x);
        Piece w;
        int partial_pieces = 0;
        while (it.next(w)) {
          const SeqGeo& s = b.seq[w.seq];
          const int item = s.item_begin + 4 * (s.n_qtiles - 1 - w.qt) + w.g;
          const int nt = nts[static_cast<size_t>(item)];
          if (w.n0 < 0 || w.n1 > nt || w.n0 >= w.n1) { ++bad; printf("balanced: bad range\n"); }
          const bool whole = w.n0 == 0 && w.n1 == nt;
          if (whole != (w.slot < 0)) { ++bad; printf("balanced: whole <-> no slot\n"); }
          if (item < head && !whole) { ++bad; printf("balanced: head item not whole\n"); }
          if (w.slot >= 0) {
            ++partial_pieces;
            if (w.slot != 2 * x && w.slot != 2 * x + 1) { ++bad; printf("balanced: foreign slot\n"); }
            if (slots[w.slot]++) { ++bad; printf("balanced: slot reused\n"); }
          }
          if (item >= head) by_item[static_cast<size_t>(item - head)].push_back({x, w.n0, w.n1, w.slot});
          for (int n = w.n0; n < w.n1; ++n) cover[static_cast<size_t>(off[static_cast<size_t>(item)] + n)]++;
        }
        if (partial_pieces > 2) { ++bad; printf("balanced: more than two partial pieces\n"); }
      }
      for (int i = 0; i < n_items; ++i)
        for (int n = 0; n < nts[static_cast<size_t>(i)]; ++n) {
          ++checks;
          if (cover[static_cast<size_t>(off[static_cast<size_t>(i)] + n)] != 1 && ++bad < 10)
            printf("balanced coverage G=%d hr=%d item=%d tile=%d\n", G, hr, i, n);
        }
      for (int k = 0; k < n_tail; ++k) {  // what the merge kernel reads
        int x_lo = 0, n = 0;
        balanced_item_pieces(tp.v, n_tail, G, k, x_lo, n);
        const std::vector<Emitted>& e = by_item[static_cast<size_t>(k)];
        ++checks;
        if (static_cast<int>(e.size()) != n) { ++bad; printf("balanced: piece count %d vs %d\n", static_cast<int>(e.size()), n); continue; }
        if (n == 1 && e[0].slot >= 0) { ++bad; printf("balanced: unsplit item wrote a slot\n"); }
        int next = 0;
        for (int i = 0; i < n; ++i) {
          if (e[static_cast<size_t>(i)].x != x_lo + i || e[static_cast<size_t>(i)].n0 != next) { ++bad; printf("balanced: piece order\n"); }
          if (n > 1 && e[static_cast<size_t>(i)].slot != balanced_slot(tp.v, n_tail, G, k, x_lo, i)) { ++bad; printf("balanced: merge slot\n"); }
          next = e[static_cast<size_t>(i)].n1;
        }
        if (next != nts[static_cast<size_t>(head + k)]) { ++bad; printf("balanced: item not complete\n"); }
      }
    }
  }
}

}  // namespace

int main() {
  static Batch b;
  const int qls[] = {1, 2, 5, 20, 21, 22, 42, 43, 127, 128, 129, 500, 512, 3072, 4096};
  const int extras[] = {0, 1, 100, 127, 128, 129, 255, 1000, 4096, 28672};
  const int grids[] = {1, 2, 3, 7, 64, 152, 1000};
  const int splits[] = {1, 2, 3, 4, 7, 16};
  // One sequence: every chunk shape of the workloads and around the tile edges.
  for (int tpi : {21, 42})
    for (int ql : qls)
      for (int ex : extras) {
        make_batch({{ql, ql + ex}}, tpi, b);
        check_batch(b, grids, 7, splits, 6);
      }
  // Batches of 2 to 12 sequences (some empty), seeded.
  uint32_t seed = 12345;
  for (int t = 0; t < 300; ++t) {
    const int n = 2 + static_cast<int>(lcg(seed) % 11);
    std::vector<std::pair<int, int>> lens;
    for (int i = 0; i < n; ++i) {
      const int ql = (lcg(seed) % 5 == 0) ? 0 : 1 + static_cast<int>(lcg(seed) % 600);
      const int kl = ql + static_cast<int>(lcg(seed) % 3000);
      lens.push_back({ql, kl > 0 ? kl : 1});
    }
    make_batch(lens, (t & 1) ? 42 : 21, b);
    if (b.n_items == 0) continue;
    check_batch(b, grids, 7, splits, 6);
  }
  printf("checks=%lld bad=%d\n", checks, bad);
  return bad != 0;
}
