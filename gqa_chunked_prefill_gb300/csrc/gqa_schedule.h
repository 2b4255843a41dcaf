// Work decomposition of one call, shared by the host planner, the attention
// kernel and the merge kernel (all three must agree unit for unit).
//
// An *item* is one query tile of one KV group that sweeps KV tiles 0 .. nt-1
// (128 keys each) up to the causal diagonal: 21 tokens (126 packed MMA rows)
// for the one-CTA kernel, 42 tokens for the CTA-pair kernel (21 per CTA).
// Items are ordered longest first — item i covers query tile
// qt = n_qtiles - 1 - i/4 and KV group g = i%4 — so consecutive items have
// (nearly) the same length.
//
// Work units are dealt to the G persistent CTAs in a snake: in round r, unit
// r*G + x goes to CTA x (r even) or G-1-x (r odd). The first head_items =
// head_rounds*G units are whole items. Every remaining ("tail") item is split
// into S pieces of equal KV length, S consecutive units: tail piece t covers
// tiles [s*nt/S, (s+1)*nt/S) of item head_items + t/S, s = t%S, and (when
// S > 1) writes a normalised FP32 partial to slot t; merge_tail_kernel then
// combines the S slots of every tail item.
//
// Why this shape: in every round all CTAs sweep the KV range of items of
// equal length from the same starting key in lockstep, so the K/V tiles in
// flight at any moment are few and stay in L2 even when the whole K/V does
// not fit; only the last, partial round is cut into pieces so that it spreads
// over all CTAs (and its pieces with the same s are aligned as well).
#pragma once

#include <cstdint>

namespace gqa {

struct Geometry {
  int q_len;         // tokens in the chunk
  int p0;            // kv_len - q_len: position of the chunk's first token
  int n_qtiles;      // ceil(q_len / tok_per_item)
  int tok_per_item;  // 21 (one CTA per item) or 42 (a CTA pair per item)
};

// KV tiles an item of query tile qt visits: keys 0 .. p0 + last token of the tile.
__host__ __device__ inline int item_tiles(const Geometry& geo, int qt) {
  const int end = (qt + 1) * geo.tok_per_item;
  const int tok_end = end < geo.q_len ? end : geo.q_len;
  return (geo.p0 + tok_end + 127) / 128;
}

struct Schedule {
  int head_items;   // items processed whole (a multiple of the grid, or all items)
  int tail_splits;  // S: pieces per tail item (1 = tail items are whole too)
  int n_units;      // head_items + (n_items - head_items) * S
};

// One unit of work: tiles [n0, n1) of item (qt, g). slot < 0: the unit is a
// whole item and writes the output directly; otherwise it writes partial slot `slot`.
struct Piece {
  int qt, g, n0, n1, slot;
};

__host__ __device__ inline Piece unit_piece(const Geometry& geo, const Schedule& sc, int u) {
  Piece w;
  int item, s = 0;
  if (u < sc.head_items) {
    item = u;
  } else {
    const int t = u - sc.head_items;
    item = sc.head_items + t / sc.tail_splits;
    s = t % sc.tail_splits;
  }
  w.qt = geo.n_qtiles - 1 - item / 4;
  w.g = item % 4;
  const int nt = item_tiles(geo, w.qt);
  if (u < sc.head_items || sc.tail_splits == 1) {
    w.n0 = 0;
    w.n1 = nt;
    w.slot = -1;
  } else {
    w.n0 = static_cast<int>(static_cast<long long>(s) * nt / sc.tail_splits);
    w.n1 = static_cast<int>(static_cast<long long>(s + 1) * nt / sc.tail_splits);
    w.slot = u - sc.head_items;
  }
  return w;
}

// Iterates one CTA's units in order; every role of the CTA runs its own copy.
struct PieceIter {
  Geometry geo;
  Schedule sc;
  int G, b, round;

  __host__ __device__ inline void init(const Geometry& g_, const Schedule& s_, int G_, int b_) {
    geo = g_;
    sc = s_;
    G = G_;
    b = b_;
    round = 0;
  }

  __host__ __device__ inline bool next(Piece& w) {
    const int u = round * G + ((round & 1) ? (G - 1 - b) : b);
    if (u >= sc.n_units) return false;
    ++round;
    w = unit_piece(geo, sc, u);  // never empty: the planner keeps S <= every tail item's tiles
    return true;
  }
};

}  // namespace gqa
