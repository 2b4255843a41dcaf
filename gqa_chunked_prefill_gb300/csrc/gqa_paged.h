// Paged K/V addressing: which cache rows the attention kernel's TMA producer
// copies for one box of keys. Shared by the kernel and the host brute-force
// check (tests/paged_rows_check.cpp).
//
// Layout (gfx936 DCU上实现INT8 QK MMAC：分页访存、Fragment映射与GQA适配, §3: a
// logical key token goes through the block table to its physical block, then
// to its slot there): the caches are [num_pages][page_size][4][256] and
// logical key j of the sequence is cache row
//     table[j / page_size] * page_size + j % page_size
// of the cache viewed as [num_pages * page_size][4][256], which is what the
// TMA tensor maps describe.
//
// A box is 64 or 128 consecutive logical keys starting at a multiple of 64.
// Inside one page it is one copy. Across pages it is cut into pieces of
// sub_rows = gcd(page_size, 64) keys: sub_rows divides both the page size and
// the box start, so no piece crosses a page. The V box of the tile that holds
// key kv_len-1 is always cut into 16-key pieces, so that only the rows past
// kv_len in its last partial piece (< 16) come from the cache's unused slots;
// the kernel zeroes those. Pieces and boxes that start at or past kv_len copy
// from oob_row, past the end of the cache, where TMA writes zeros; the block
// table is never read past its ceil(kv_len / page_size) entries.
#pragma once

// Unroll hint for the CUDA compiler only (the host brute-force check builds
// this header with a plain C++ compiler).
#if defined(__CUDACC__)
#define GQA_UNROLL _Pragma("unroll")
#else
#define GQA_UNROLL
#endif

namespace gqa {

struct PagedGeom {
  int kv_len;
  int page_size;  // a multiple of 16
  int num_pages;
  int sub_rows;   // gcd(page_size, 64): 16, 32 or 64
  int oob_row;    // num_pages * page_size
};

struct PagedRun {
  int n;       // 0: one copy of the whole box at row[0]; else n pieces of `sub` rows
  int sub;     // rows per piece (the box's rows when n == 0)
  int row[8];  // cache row where the box / each piece starts
  bool bad;    // a block-table entry outside [0, num_pages) was met (read as zeros)
};

// The common case of map_paged_run, kept apart so that a kernel can inline it
// and call the rest out of line: true when the box is one copy — it starts at
// or past kv_len (row = oob_row) or lies inside one page (row = its cache row,
// or oob_row with *bad set if that page's entry is outside the cache).
template <typename Read>
__host__ __device__ inline bool paged_whole_box(const PagedGeom& g, int r0, int rows, bool v_fix,
                                                Read&& read, int* row, bool* bad) {
  *row = g.oob_row;
  *bad = false;
  if (r0 >= g.kv_len) return true;  // the whole box lies past the sequence: zero fill
  const int pg0 = r0 / g.page_size;
  const int off0 = r0 - pg0 * g.page_size;
  if (v_fix || off0 + rows > g.page_size) return false;
  const int e = read(pg0);
  if (e >= 0 && e < g.num_pages) *row = e * g.page_size + off0;
  else *bad = true;
  return true;
}

// Maps the box of `rows` keys (64 or 128) that starts at logical key r0.
// `read(pg)` returns block-table entry pg; it is called only for pages that
// hold a key below kv_len.
template <typename Read>
__host__ __device__ inline void map_paged_run(const PagedGeom& g, int r0, int rows, bool v_fix,
                                              Read&& read, PagedRun& run) {
  run.n = 0;
  run.sub = rows;
  if (paged_whole_box(g, r0, rows, v_fix, read, &run.row[0], &run.bad)) return;
  const int pg0 = r0 / g.page_size;
  const int off0 = r0 - pg0 * g.page_size;
  run.sub = v_fix ? 16 : g.sub_rows;
  run.n = rows / run.sub;
  int ent[8];
  unsigned live = 0;  // pieces that start below kv_len
  int pg = pg0, off = off0;
  GQA_UNROLL
  for (int i = 0; i < 8; ++i) {  // independent block-table reads, issued together
    run.row[i] = off;
    ent[i] = 0;
    if (i < run.n && r0 + i * run.sub < g.kv_len) {
      ent[i] = read(pg);
      live |= 1u << i;
    }
    off += run.sub;
    if (off == g.page_size) {
      off = 0;
      ++pg;
    }
  }
  GQA_UNROLL
  for (int i = 0; i < 8; ++i) {
    const bool is_live = (live >> i) & 1u;
    const bool in_cache = ent[i] >= 0 && ent[i] < g.num_pages;
    if (is_live && !in_cache) run.bad = true;
    run.row[i] = is_live && in_cache ? run.row[i] + ent[i] * g.page_size : g.oob_row;
  }
}

}  // namespace gqa
