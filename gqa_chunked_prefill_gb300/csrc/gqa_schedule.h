// Work decomposition of one call, shared by the host planner, the attention
// kernel and the merge kernel (all three must agree tile for tile).
//
// An *item* is one 21-token query tile of one KV group: 126 packed MMA rows
// that sweep KV tiles 0 .. nt-1 (128 keys each) up to the causal diagonal.
// Items are ordered longest first — rank r = 0 is the last query tile (it
// sees the most keys) — and the 4 KV groups of a query tile are consecutive:
// item i = 4 r + g covers query tile qt = n_qtiles - 1 - r.
//
// Two schedules over a persistent grid of G CTAs:
//  * kScheduleItems: whole items, CTA b takes items b, 2G-1-b, 2G+b, ... (a
//    snake over the longest-first order). No item is split, no merge pass.
//  * kScheduleRanges: the items' KV tiles are laid end to end (W tiles in
//    all) and CTA b takes the contiguous range [bW/G, (b+1)W/G). An item cut
//    by a range boundary is computed in pieces by consecutive CTAs; a piece
//    that does not start at the item's first tile goes to partial slot 2b,
//    one that starts there but stops early goes to slot 2b+1, and
//    merge_ranges_kernel combines the pieces of every cut item.
#pragma once

#include <cstdint>

namespace gqa {

constexpr int kScheduleItems = 0;
constexpr int kScheduleRanges = 1;

struct Geometry {
  int q_len;     // tokens in the chunk
  int p0;        // kv_len - q_len: position of the chunk's first token
  int n_qtiles;  // ceil(q_len / 21)
};

// KV tiles an item of query tile qt visits: keys 0 .. p0 + last token of the tile.
__host__ __device__ inline int item_tiles(const Geometry& geo, int qt) {
  const int tok_end = (qt + 1) * 21 < geo.q_len ? (qt + 1) * 21 : geo.q_len;
  return (geo.p0 + tok_end + 127) / 128;
}

// sum_{i=0}^{n-1} floor((a*i + b) / m) for n, a, b >= 0, m > 0, by the usual
// Euclid-like reduction: strip the integer parts of a/m and b/m, then count
// the lattice points under the remaining line with the roles of a and m swapped.
__host__ __device__ inline long long floor_sum(long long n, long long m, long long a, long long b) {
  long long ans = 0;
  while (n > 0) {
    if (a >= m) {
      ans += (n - 1) * n / 2 * (a / m);
      a %= m;
    }
    if (b >= m) {
      ans += n * (b / m);
      b %= m;
    }
    const long long y_max = a * n + b;
    if (y_max < m) break;
    n = y_max / m;
    b = y_max % m;
    const long long t = m;
    m = a;
    a = t;
  }
  return ans;
}

// Tiles of query tiles 0 .. x-1 of one KV group (x <= n_qtiles). Every tile but
// the last holds 21 tokens, so nt(qt) = floor((p0 + 21 qt + 21 + 127) / 128).
__host__ __device__ inline long long tiles_below(const Geometry& geo, int x) {
  const int full = x < geo.n_qtiles - 1 ? x : geo.n_qtiles - 1;
  long long s = full > 0 ? floor_sum(full, 128, 21, geo.p0 + 21 + 127) : 0;
  if (x == geo.n_qtiles && x > 0) s += item_tiles(geo, geo.n_qtiles - 1);
  return s;
}

// Total KV tiles over all items (all 4 groups).
__host__ __device__ inline long long total_tiles(const Geometry& geo) {
  return 4 * tiles_below(geo, geo.n_qtiles);
}

// First global tile of the items of rank r (group 0), given tiles_below(n_qtiles).
__host__ __device__ inline long long rank_start(const Geometry& geo, int r, long long t_all) {
  return 4 * (t_all - tiles_below(geo, geo.n_qtiles - r));
}

struct ItemPos {
  int r, g;         // rank and KV group
  int nt;           // tiles of the item
  long long start;  // its first global tile
};

// The item holding global tile t (0 <= t < total_tiles).
__host__ __device__ inline ItemPos locate(const Geometry& geo, long long t) {
  const long long t_all = tiles_below(geo, geo.n_qtiles);
  int lo = 0, hi = geo.n_qtiles - 1;  // largest r with rank_start(r) <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    if (rank_start(geo, mid, t_all) <= t) lo = mid; else hi = mid - 1;
  }
  ItemPos p;
  p.r = lo;
  p.nt = item_tiles(geo, geo.n_qtiles - 1 - lo);
  const long long rs = rank_start(geo, lo, t_all);
  p.g = static_cast<int>((t - rs) / p.nt);
  p.start = rs + static_cast<long long>(p.g) * p.nt;
  return p;
}

// First global tile of CTA b's range under kScheduleRanges.
__host__ __device__ inline long long range_lo(long long W, int G, int b) {
  return W * b / G;
}

// The CTA whose range holds global tile x.
__host__ __device__ inline int range_owner(long long W, int G, long long x) {
  return static_cast<int>(((x + 1) * G + W - 1) / W - 1);
}

// One piece of work of a CTA: tiles [n0, n1) of item (qt, g); slot < 0 means the
// piece is the whole item and writes the output directly.
struct Piece {
  int qt, g, n0, n1, slot;
};

// Iterates one CTA's pieces in order; every role of the CTA runs its own copy.
struct PieceIter {
  Geometry geo;
  int mode, G, b;
  // kScheduleItems
  int round;
  int n_items;
  // kScheduleRanges
  long long t, hi;
  ItemPos cur;

  __host__ __device__ inline void init(const Geometry& g_, int mode_, int G_, int b_, long long W) {
    geo = g_;
    mode = mode_;
    G = G_;
    b = b_;
    round = 0;
    n_items = 4 * geo.n_qtiles;
    t = hi = 0;
    if (mode == kScheduleRanges) {
      t = range_lo(W, G, b);
      hi = range_lo(W, G, b + 1);
      if (t < hi) cur = locate(geo, t);
    }
  }

  __host__ __device__ inline bool next(Piece& w) {
    if (mode == kScheduleItems) {
      const int u = round * G + ((round & 1) ? (G - 1 - b) : b);
      if (u >= n_items) return false;
      ++round;
      w.qt = geo.n_qtiles - 1 - u / 4;
      w.g = u % 4;
      w.n0 = 0;
      w.n1 = item_tiles(geo, w.qt);
      w.slot = -1;
      return true;
    }
    if (t >= hi) return false;
    const long long n0 = t - cur.start;
    const long long n1 = (hi - cur.start) < cur.nt ? (hi - cur.start) : cur.nt;
    w.qt = geo.n_qtiles - 1 - cur.r;
    w.g = cur.g;
    w.n0 = static_cast<int>(n0);
    w.n1 = static_cast<int>(n1);
    w.slot = n0 > 0 ? 2 * b : (n1 < cur.nt ? 2 * b + 1 : -1);
    t = cur.start + n1;
    if (n1 == cur.nt) {  // move to the next item
      cur.start += cur.nt;
      if (++cur.g == 4) {
        cur.g = 0;
        ++cur.r;
        if (cur.r < geo.n_qtiles) cur.nt = item_tiles(geo, geo.n_qtiles - 1 - cur.r);
      }
    }
    return true;
  }
};

}  // namespace gqa
