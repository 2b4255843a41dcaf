// Host check of the paged K/V addressing in gqa_paged.h (compiled with g++ by
// tests/test_paged_cpu.py). For many page sizes, sequence lengths and seeded
// block tables (a permutation of the cache's pages, optionally with entries
// outside the cache) it maps every box the attention kernel's TMA producer
// loads — one-CTA K (128 keys) and V (2 x 64 keys), CTA-pair K (2 x 64 keys)
// and V (128 keys), for every KV tile of the sequence and one past it — and
// checks, key by key:
//  * a key below kv_len whose page entry is valid is copied from cache row
//    table[j / page_size] * page_size + j % page_size;
//  * a key below kv_len on an invalid entry, and every key of a box or piece
//    that starts at or past kv_len, is copied from a row past the cache
//    (TMA zero fill), and an invalid entry sets `bad`;
//  * in the V box of the tile holding key kv_len-1, every key from the next
//    multiple of 16 above kv_len on reads zeros (the kernel zeroes the rest);
//  * V boxes of earlier tiles hold only keys below kv_len;
//  * no copy crosses a page or runs past the cache's end; pieces tile the box
//    exactly (n * sub == rows, n <= 8, sub the documented size);
//  * the block table is never read at or past ceil(kv_len / page_size).
// Prints "checks=N bad=M" and exits non-zero on any mismatch.
#include "gqa_paged.h"

#include <cstdint>
#include <cstdio>
#include <vector>

using namespace gqa;

namespace {

uint32_t lcg(uint32_t& s) {
  s = s * 1664525u + 1013904223u;
  return s >> 8;
}

int gcd(int a, int b) { return b == 0 ? a : gcd(b, a % b); }

}  // namespace

int main() {
  long long checks = 0;
  int bad = 0;
  auto fail = [&](const char* what, int ps, int kv, int r0, int rows, int i) {
    if (bad < 20)
      std::printf("FAIL %s: page %d kv_len %d box r0 %d rows %d key %d\n", what, ps, kv, r0, rows,
                  r0 + i);
    ++bad;
  };
  const int page_sizes[] = {16, 32, 48, 64, 80, 96, 112, 128, 144, 192, 256, 784, 1024, 4096};
  const int kv_lens[] = {1,   2,   15,  16,  17,   31,   63,   64,   65,  127, 128,
                         129, 191, 255, 256, 257,  300,  783,  784,  785, 1000, 1568,
                         2047, 2048, 4097, 8191, 8192, 32768};
  for (int ps : page_sizes)
    for (int kv : kv_lens)
      for (int mode = 0; mode < 2; ++mode) {  // 0: valid table; 1: some entries outside the cache
        const int n_log = (kv + ps - 1) / ps;
        const int num_pages = n_log + 3;
        uint32_t seed = 977u * ps + 31u * kv + mode;
        std::vector<int> perm(num_pages);
        for (int i = 0; i < num_pages; ++i) perm[i] = i;
        for (int i = num_pages - 1; i > 0; --i) {
          const int j = static_cast<int>(lcg(seed) % static_cast<uint32_t>(i + 1));
          const int t = perm[i];
          perm[i] = perm[j];
          perm[j] = t;
        }
        std::vector<int> table(perm.begin(), perm.begin() + n_log);
        if (mode == 1)
          for (int i = 0; i < n_log; ++i)
            if (lcg(seed) % 4 == 0) table[i] = (lcg(seed) & 1) ? -1 - i : num_pages + i;
        const PagedGeom g{kv, ps, num_pages, gcd(ps, 64), num_pages * ps};
        const int last_tile = (kv - 1) / 128;
        const int v_fix_tile = kv % 128 ? last_tile : -1;
        bool read_past = false;
        auto read = [&](int pg) {
          if (pg < 0 || pg >= n_log) {
            read_past = true;
            return 0;
          }
          return table[pg];
        };
        struct Box {
          int off, rows;
          bool is_v;
        };
        const Box boxes[] = {{0, 128, false}, {0, 64, true},  {64, 64, true},
                             {0, 64, false},  {64, 64, false}, {0, 128, true}};
        for (int n = 0; n <= last_tile + 1; ++n)
          for (const Box& b : boxes) {
            const int r0 = n * 128 + b.off;
            const bool v_fix = b.is_v && n == v_fix_tile;
            PagedRun run;
            read_past = false;
            map_paged_run(g, r0, b.rows, v_fix, read, run);
            ++checks;
            if (read_past) fail("block table read past its end", ps, kv, r0, b.rows, 0);
            bool saw_bad = false;
            if (run.n == 0) {
              if (run.sub != b.rows) fail("whole box size", ps, kv, r0, b.rows, 0);
              if (run.row[0] < g.oob_row && run.row[0] % ps + b.rows > ps)
                fail("box crosses a page", ps, kv, r0, b.rows, 0);
            } else {
              const int want_sub = v_fix ? 16 : g.sub_rows;
              if (run.sub != want_sub || run.n * run.sub != b.rows || run.n > 8)
                fail("piece sizes", ps, kv, r0, b.rows, 0);
              for (int p = 0; p < run.n; ++p)
                if (run.row[p] < g.oob_row && run.row[p] % ps + run.sub > ps)
                  fail("piece crosses a page", ps, kv, r0, b.rows, p * run.sub);
            }
            if (b.is_v && n < last_tile + 1 && !v_fix && r0 + b.rows > kv)
              fail("V box past kv_len outside the last tile", ps, kv, r0, b.rows, 0);
            const int piece = run.n == 0 ? b.rows : run.sub;
            for (int i = 0; i < b.rows; ++i) {
              const int j = r0 + i;
              const int start = run.row[run.n == 0 ? 0 : i / run.sub];
              const int src = start + i % piece;
              const int piece_key0 = r0 + (i / piece) * piece;
              ++checks;
              if (start >= g.oob_row) {
                // zero fill: fine unless a valid key below kv_len needed real data
                if (j < kv) {
                  const int e = table[j / ps];
                  if (e >= 0 && e < num_pages) fail("valid key read as zero", ps, kv, r0, b.rows, i);
                  else saw_bad = true;
                }
                continue;
              }
              if (piece_key0 >= kv) fail("piece past kv_len not zero-filled", ps, kv, r0, b.rows, i);
              if (j < kv) {
                const int e = table[j / ps];
                if (!(e >= 0 && e < num_pages)) fail("invalid entry followed", ps, kv, r0, b.rows, i);
                else if (src != e * ps + j % ps) fail("wrong cache row", ps, kv, r0, b.rows, i);
              } else if (v_fix && j >= ((kv + 15) & ~15)) {
                fail("v tail row above the 16-key boundary not zero", ps, kv, r0, b.rows, i);
              }
              if (src >= g.oob_row) fail("copy runs past the cache", ps, kv, r0, b.rows, i);
            }
            if (saw_bad != run.bad) fail("bad flag", ps, kv, r0, b.rows, 0);
          }
      }
  std::printf("checks=%lld bad=%d\n", checks, bad);
  return bad == 0 ? 0 : 1;
}
