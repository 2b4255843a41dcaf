// Work decomposition of one call, shared by the host planner, the attention
// kernel and the merge kernel (all three must agree unit for unit).
//
// A call holds one or more sequences (up to kMaxSeqs). In each, the q_len new
// tokens are the last q_len of its kv_len keys (bottom-right causal
// alignment); its rows sit at q_start of the packed Q / out / LSE and, for
// dense K/V, at kv_start of the packed K / V.
//
// An *item* is one query tile of one KV group of one sequence that sweeps KV
// tiles 0 .. nt-1 (128 keys each) up to the causal diagonal: 21 tokens (126
// packed MMA rows) for the one-CTA kernel, 42 tokens for the CTA-pair kernel
// (21 per CTA). A sequence's items are ordered longest first — item li covers
// query tile qt = n_qtiles - 1 - li/4 and KV group g = li%4 — and the host
// orders the sequences by their longest item, so the call's item list runs
// (nearly) longest first; item i belongs to the last sequence whose
// item_begin <= i.
//
// Work units are dealt to the G persistent CTAs in a snake: in round r, unit
// r*G + x goes to CTA x (r even) or G-1-x (r odd). The first head_items =
// head_rounds*G units are whole items. The remaining ("tail") items are cut in
// one of two ways:
//  - uniform (S >= 1): every tail item is split into S pieces of equal KV
//    length, S consecutive units: tail piece t covers tiles [s*nt/S,
//    (s+1)*nt/S) of item head_items + t/S, s = t%S, and (when S > 1) writes a
//    normalised FP32 partial to slot t;
//  - balanced (S = 0): the tail items' tiles are laid end to end (W of them,
//    prefix sums in a TailPrefix) and CTA x takes the range [x*W/G,
//    (x+1)*W/G), cut at item boundaries. A piece that is a whole item writes
//    the output; of the others, the CTA's first piece writes slot 2x and its
//    last piece slot 2x+1 (a range holds at most those two partial pieces).
//    Every CTA gets the same number of tiles, whatever the tail's item count.
// The merge pass (merge_tail_kernel, or merge_wide_kernel for items of 16 or more
// pieces) then combines the pieces of every split tail item.
//
// Why this shape: in every round all CTAs sweep the KV range of items of
// (nearly) equal length from the same starting key in lockstep, so the K/V
// tiles in flight at any moment are few and stay in L2 even when the whole
// K/V does not fit; only the last, partial round is cut into pieces so that it
// spreads over all CTAs (and its pieces with the same s are aligned as well).
#pragma once

#include <cstdint>

namespace gqa {

constexpr int kMaxSeqs = 128;  // sequences per call

struct SeqGeo {
  int q_start;     // first row of the sequence in the packed Q / out / LSE
  int q_len;       // its new tokens (> 0: the host leaves empty sequences out)
  int kv_start;    // first key row in the packed K / V (dense K/V; 0 when paged)
  int kv_len;      // its keys, q_len of them the new tokens' own
  int n_qtiles;    // ceil(q_len / tok_per_item)
  int item_begin;  // items of the sequences before it in the call's order
  int src;         // its index in the caller's batch (block-table row of paged K/V)
  int ks_start;    // FP8 QK^T with dense K: column of its first key in the key-scale rows
                   //   (a multiple of 4: TMA needs 16-byte-aligned starts)
};

struct Batch {
  int n_seq;
  int tok_per_item;  // 21 (one CTA per item) or 42 (a CTA pair per item)
  int n_items;       // items of the whole call
  SeqGeo seq[kMaxSeqs];
};

// KV tiles an item of query tile qt visits: keys 0 .. p0 + last token of the tile.
__host__ __device__ inline int item_tiles(const SeqGeo& s, int tpi, int qt) {
  const int end = (qt + 1) * tpi;
  const int tok_end = end < s.q_len ? end : s.q_len;
  return (s.kv_len - s.q_len + tok_end + 127) / 128;
}

struct Schedule {
  int head_items;   // items processed whole (a multiple of the grid, or all items)
  int tail_splits;  // S: pieces per tail item (1 = tail items are whole too); 0: balanced
  int n_units;      // uniform: head_items + (n_items - head_items) * S
  int n_tail;       // balanced: n_items - head_items (<= kMaxBalancedTail)
};

// Balanced tail: v[k] = KV tiles of tail items 0 .. k-1 (item head_items + k),
// k = 0 .. n_tail; v[n_tail] = W, the tail's tiles, at least the grid's G
// workers (so that no worker's range is empty) and below 2^31.
constexpr int kMaxBalancedTail = 512;
struct TailPrefix {
  int v[kMaxBalancedTail + 1];
};

// First tile of worker x's balanced-tail range (x = G: the end of the tail).
__host__ __device__ inline long long tail_range_begin(int x, long long W, int G) {
  return static_cast<long long>(x) * W / G;
}

// The worker whose balanced-tail range holds tile t (0 <= t < W): the largest x
// with x*W/G <= t, i.e. x*W < (t+1)*G.
__host__ __device__ inline int tail_worker_at(long long t, long long W, int G) {
  return static_cast<int>(((t + 1) * G + W - 1) / W) - 1;
}

// The tail item holding tile t of the balanced tail: the largest k with v[k] <= t.
__host__ __device__ inline int tail_item_at(const int* v, int n_tail, long long t) {
  int lo = 0, hi = n_tail - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (v[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Balanced tail, merge side: the pieces of tail item k are those of workers
// x_lo .. x_lo + n - 1 (n = 1: the item was not split). Piece i's slot is
// merge_slot(...): the first worker may have started in an earlier item, so
// its piece of item k is its last one (slot 2x+1); every later worker's range
// starts inside item k, so the piece is its first one (slot 2x).
__host__ __device__ inline void balanced_item_pieces(const int* v, int n_tail, int G, int k,
                                                     int& x_lo, int& n) {
  const long long W = v[n_tail];
  x_lo = tail_worker_at(v[k], W, G);
  n = tail_worker_at(static_cast<long long>(v[k + 1]) - 1, W, G) - x_lo + 1;
}
__host__ __device__ inline int balanced_slot(const int* v, int n_tail, int G, int k, int x_lo,
                                             int i) {
  if (i > 0) return 2 * (x_lo + i);
  return 2 * x_lo + (tail_range_begin(x_lo, v[n_tail], G) < v[k] ? 1 : 0);
}

// Item i of the call: its sequence, query tile and KV group.
__host__ __device__ inline void item_of(const Batch& b, int i, int& seq, int& qt, int& g) {
  int lo = 0, hi = b.n_seq - 1;  // the last sequence with item_begin <= i
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (b.seq[mid].item_begin <= i) lo = mid;
    else hi = mid - 1;
  }
  seq = lo;
  const int li = i - b.seq[lo].item_begin;
  qt = b.seq[lo].n_qtiles - 1 - li / 4;
  g = li % 4;
}

// One unit of work: tiles [n0, n1) of item (seq, qt, g). slot < 0: the unit is
// a whole item and writes the output directly; otherwise it writes partial slot
// `slot`. tail: the item's index among the tail items (item - head_items), or -1
// for an item of the whole rounds.
struct Piece {
  int seq, qt, g, n0, n1, slot, tail;
};

// Pieces of tail item j and where piece s (KV order) wrote its partial, for
// either cut (S = sc.tail_splits; S == 0: balanced, from the prefix sums v over
// G workers). n < 2: the item was not split.
__host__ __device__ inline int tail_item_pieces(const Schedule& sc, const int* v, int G, int j,
                                                int& x_lo) {
  x_lo = 0;
  if (sc.tail_splits > 0) return sc.tail_splits;
  int n;
  balanced_item_pieces(v, sc.n_tail, G, j, x_lo, n);
  return n;
}
__host__ __device__ inline int tail_piece_slot(const Schedule& sc, const int* v, int G, int j,
                                               int x_lo, int s) {
  return sc.tail_splits > 0 ? j * sc.tail_splits + s : balanced_slot(v, sc.n_tail, G, j, x_lo, s);
}

__host__ __device__ inline Piece unit_piece(const Batch& b, const Schedule& sc, int u) {
  Piece w;
  int item, s = 0;
  if (u < sc.head_items) {
    item = u;
  } else {
    const int t = u - sc.head_items;
    item = sc.head_items + t / sc.tail_splits;
    s = t % sc.tail_splits;
  }
  item_of(b, item, w.seq, w.qt, w.g);
  w.tail = u < sc.head_items ? -1 : item - sc.head_items;
  const int nt = item_tiles(b.seq[w.seq], b.tok_per_item, w.qt);
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
  const Batch* b;
  const int* tail;  // balanced tail: the TailPrefix values (unused otherwise)
  Schedule sc;
  int G, x, round;
  int k;                      // balanced tail: -1 before it, then the tail item at `pos`
  long long pos, begin, end;  // balanced tail: next tile, this worker's range

  __host__ __device__ inline void init(const Batch* b_, const int* tail_, const Schedule& s_,
                                       int G_, int x_) {
    b = b_;
    tail = tail_;
    sc = s_;
    G = G_;
    x = x_;
    round = 0;
    k = -1;
    pos = begin = end = 0;
  }

  __host__ __device__ inline bool next(Piece& w) {
    if (k < 0) {
      const int u = round * G + ((round & 1) ? (G - 1 - x) : x);
      if (sc.tail_splits > 0 ? u < sc.n_units : u < sc.head_items) {
        ++round;
        w = unit_piece(*b, sc, u);  // never empty: the planner keeps S <= every item's tiles
        return true;
      }
      if (sc.tail_splits > 0) return false;
      if (sc.n_tail < 1) return false;
      const long long W = tail[sc.n_tail];
      begin = pos = tail_range_begin(x, W, G);
      end = tail_range_begin(x + 1, W, G);
      k = tail_item_at(tail, sc.n_tail, pos);
    }
    if (pos >= end) return false;
    const long long s = tail[k], e = tail[k + 1];
    const long long stop = end < e ? end : e;
    item_of(*b, sc.head_items + k, w.seq, w.qt, w.g);
    w.tail = k;
    w.n0 = static_cast<int>(pos - s);
    w.n1 = static_cast<int>(stop - s);
    w.slot = (pos == s && stop == e) ? -1 : 2 * x + (pos == begin ? 0 : 1);
    pos = stop;
    ++k;
    return true;
  }
};

}  // namespace gqa
