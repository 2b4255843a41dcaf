// Host side of libgqa_prefill.so: the C ABI declared in include/gqa_prefill.h.
//
// Responsibilities: validate the call and refuse unsupported shapes (the
// dedicated kernel of DCU使用技术报告（中篇）, §2 only takes one BF16 sequence
// with 24Q/4KV/d256 and sends everything else away; the INT8 QK MMAC page, §7,
// rejects wrong layouts rather than mapping them silently), plan the work from
// the real q_len/kv_len of this chunk (same report §3 dispatches on the
// kernel's actual q_len and kv_len, not on a dataset bucket), encode the TMA
// tensor maps, allocate split partials in stream order, and launch.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include <cudaTypedefs.h>

#include "gqa_internal.h"
#include "gqa_prefill.h"
#include "gqa_schedule.h"

namespace gqa {
namespace {

static_assert(kMaxSeqs == GQA_MAX_SEQS, "the sequence table and the public limit must agree");
constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s per device-side wait

// ------------------------------------------------------------------ planner --
// Cost model in units of one 128-key KV tile of one item (QK^T + PV of a
// 128 x 128 x 256 block per CTA: ~1.3 us of tensor-core time on one SM at peak).
constexpr int64_t kPieceOverheadTiles = 2;   // Q load, pipeline fill, epilogue
constexpr double kTileUs = 1.5;              // planning estimate per tile, one-CTA kernel
// Per tile of a CTA pair (the same work per SM as a one-CTA tile). Measured on
// GB300 the pair kernel is ~1.1x faster per tile (4096x32768: 1.75 ms vs
// 1.92 ms; 3072x16384: 0.67 ms vs 0.74 ms): each SM streams half the operands.
constexpr double kPairTileUs = 1.35;
// Paged K/V: against dense K/V the one-CTA kernel's launch takes 13 % longer at
// 1024-key pages, 30 % at 784 and up to 2x at 16 (512x32768), the pair's 0-5 %
// at 1024 and 784 (each SM brings in half of every tile, and the paged boxes'
// extra copies and block-table reads cost it less). Paged calls weigh the
// one-CTA plan's estimate by this factor; measured, the pair then won on every
// paged shape tried (512x32768, 512x4096, 3072x16384; pages 16 to 1024).
constexpr double kPagedOneCtaFactor = 1.25;
constexpr double kMergeBytesPerUs = 6.0e6;   // effective bandwidth of the merge pass (partials in L2)
constexpr double kMergeLaunchUs = 3.0;       // its launch, mostly hidden by programmatic launch
constexpr int64_t kPartialRowBytes = (kHeadDim + 1) * 4;  // FP32 O row + base-2 LSE
constexpr int kSplitCandidates[] = {1, 2, 3, 4, 5, 6, 8, 10, 12, 16, 24, 32};
constexpr int kForceBalanced = GQA_FORCE_BALANCED_TAIL;  // force_splits value: balanced tail

// One sequence of a call as the caller gives it: its rows in the packed Q /
// out / LSE and (dense K/V) K / V.
struct SeqIn {
  int q_start, q_len, kv_start, kv_len;
  int ks_start;  // FP8 QK^T, dense K: first key-scale column (see key_scale_starts)
};

// Key-scale columns of a dense FP8 batch: sequence b's scales start at the sum of
// its predecessors' kv_len, each rounded up to a multiple of 4, so that every
// tile's scales start on 16 bytes (a TMA requirement). Returns the columns used.
int64_t key_scale_starts(std::vector<SeqIn>* seqs) {
  int64_t col = 0;
  for (SeqIn& s : *seqs) {
    s.ks_start = static_cast<int>(col);
    col += (static_cast<int64_t>(s.kv_len) + 3) / 4 * 4;
  }
  return col;
}

int tok_per_item(int variant) { return variant == 2 ? 2 * kTokPerTile : kTokPerTile; }

// The call's sequence table for `variant`: empty sequences left out, the rest
// ordered by their longest item (longest first; ties keep the caller's order),
// with the items of the sequences before each one counted in item_begin.
void build_batch(const std::vector<SeqIn>& in, int variant, Batch* b) {
  const int tpi = tok_per_item(variant);
  std::vector<int> idx;
  std::vector<int> longest(in.size(), 0);
  for (size_t i = 0; i < in.size(); ++i) {
    if (in[i].q_len <= 0) continue;
    idx.push_back(static_cast<int>(i));
    const SeqGeo g{0, in[i].q_len, 0, in[i].kv_len, (in[i].q_len + tpi - 1) / tpi, 0, 0, 0};
    longest[i] = item_tiles(g, tpi, g.n_qtiles - 1);
  }
  std::stable_sort(idx.begin(), idx.end(), [&](int a, int c) { return longest[a] > longest[c]; });
  b->n_seq = static_cast<int>(idx.size());
  b->tok_per_item = tpi;
  int items = 0;
  for (size_t k = 0; k < idx.size(); ++k) {
    const SeqIn& s = in[static_cast<size_t>(idx[k])];
    const int n_qtiles = (s.q_len + tpi - 1) / tpi;
    b->seq[k] = SeqGeo{s.q_start, s.q_len, s.kv_start, s.kv_len, n_qtiles, items, idx[k],
                       s.ks_start};
    items += kKvHeads * n_qtiles;
  }
  b->n_items = items;
}

// KV tiles of every item of the call, in the call's item order.
std::vector<int> item_tile_counts(const Batch& b) {
  std::vector<int> t(static_cast<size_t>(b.n_items));
  for (int i = 0; i < b.n_items; ++i) {
    int seq, qt, g;
    item_of(b, i, seq, qt, g);
    t[static_cast<size_t>(i)] = item_tiles(b.seq[seq], b.tok_per_item, qt);
  }
  return t;
}

// Fills *plan for `variant` (1: one CTA per item, 2: a CTA pair per item) with
// head_rounds whole rounds and S-way tail splits over `workers` CTAs (or
// pairs), simulating the snake deal of gqa_schedule.h over the items' tile
// counts; S must not exceed the shortest item's tiles. Returns the estimated
// time in us.
double plan_schedule(const std::vector<int>& tiles, int q_tiles, int num_sms, int variant,
                     int workers, int head_rounds, int S, gqa_prefill_plan* plan) {
  const int n_items = static_cast<int>(tiles.size());
  const int cpi = variant == 2 ? 2 : 1;
  const int head = std::min(head_rounds * workers, n_items);
  const int n_units = head + (n_items - head) * S;
  workers = std::max(1, std::min(workers, n_units));
  std::vector<int64_t> load(static_cast<size_t>(workers), 0);
  int64_t total = 0;
  for (int u = 0; u < n_units; ++u) {
    const int r = u / workers, x = u % workers;
    const int b = (r & 1) ? workers - 1 - x : x;
    int len;
    if (u < head) {
      len = tiles[static_cast<size_t>(u)];
    } else {
      const int t = u - head, s = t % S;
      const int64_t nt = tiles[static_cast<size_t>(head + t / S)];
      len = static_cast<int>((s + 1) * nt / S - s * nt / S);
    }
    load[static_cast<size_t>(b)] += len + kPieceOverheadTiles;
    total += len;
  }
  const int tail = n_items - head;
  const bool split = S > 1 && tail > 0;
  std::memset(plan, 0, sizeof(*plan));
  plan->num_sms = num_sms;
  plan->q_tiles = q_tiles;
  plan->n_items = n_items;
  plan->head_rounds = head / workers;
  plan->tail_items = tail;
  plan->tail_splits = S;
  plan->n_units = n_units;
  plan->grid = workers * cpi;
  plan->kernels_per_call = split ? 2 : 1;
  plan->variant = variant;
  plan->total_tiles = total;
  plan->workspace_bytes =
      split ? static_cast<int64_t>(tail) * S * cpi * kRowsPerTile * kPartialRowBytes : 0;
  plan->est_makespan_tiles = *std::max_element(load.begin(), load.end());
  double us = static_cast<double>(plan->est_makespan_tiles) * (variant == 2 ? kPairTileUs : kTileUs);
  if (split) {
    const double bytes =
        tail * static_cast<double>(cpi * kRowsPerTile) * (S * kPartialRowBytes + 520.0);
    us += bytes / kMergeBytesPerUs + kMergeLaunchUs;
  }
  return us;
}

// Fills *plan for `variant` with head_rounds whole rounds and a balanced tail
// (gqa_schedule.h): every worker takes an equal share of the remaining items'
// tiles, cut at item boundaries. Returns the estimated time in us, or a
// negative value when the tail does not fit the balanced form (no tail item,
// more than kMaxBalancedTail of them, fewer tiles than workers, or 2^31 tiles
// and more). Without whole rounds the grid shrinks to the tail's tile count.
double plan_balanced(const std::vector<int>& tiles, int q_tiles, int num_sms, int variant,
                     int workers, int head_rounds, gqa_prefill_plan* plan) {
  const int n_items = static_cast<int>(tiles.size());
  const int cpi = variant == 2 ? 2 : 1;
  const int head = std::min(head_rounds * workers, n_items);
  const int n_tail = n_items - head;
  if (n_tail < 1 || n_tail > kMaxBalancedTail) return -1.0;
  std::vector<int64_t> prefix(static_cast<size_t>(n_tail) + 1, 0);
  for (int k = 0; k < n_tail; ++k)
    prefix[static_cast<size_t>(k) + 1] = prefix[static_cast<size_t>(k)] + tiles[static_cast<size_t>(head + k)];
  const int64_t W = prefix[static_cast<size_t>(n_tail)];
  if (head == 0) workers = static_cast<int>(std::min<int64_t>(workers, W));
  if (W < workers || W > INT32_MAX) return -1.0;
  std::vector<int64_t> load(static_cast<size_t>(workers), 0);
  int64_t total = W;
  for (int u = 0; u < head; ++u) {  // whole rounds: the snake deal
    const int r = u / workers, x = u % workers;
    const int b = (r & 1) ? workers - 1 - x : x;
    load[static_cast<size_t>(b)] += tiles[static_cast<size_t>(u)] + kPieceOverheadTiles;
    total += tiles[static_cast<size_t>(u)];
  }
  int pieces = 0, partial = 0, split_items = 0;
  int k = 0;
  for (int x = 0; x < workers; ++x) {
    const int64_t a = x * W / workers, e = (x + 1) * W / workers;
    load[static_cast<size_t>(x)] += e - a;
    while (prefix[static_cast<size_t>(k) + 1] <= a) ++k;
    for (int64_t pos = a; pos < e; ++k) {
      const int64_t s = prefix[static_cast<size_t>(k)], f = prefix[static_cast<size_t>(k) + 1];
      const int64_t stop = std::min(e, f);
      ++pieces;
      if (pos != s || stop != f) ++partial;
      if (pos == s && stop != f) ++split_items;  // counted once: at the item's first piece
      load[static_cast<size_t>(x)] += kPieceOverheadTiles;
      pos = stop;
      if (stop < f) break;  // the item continues in the next worker's range
    }
  }
  std::memset(plan, 0, sizeof(*plan));
  plan->num_sms = num_sms;
  plan->q_tiles = q_tiles;
  plan->n_items = n_items;
  plan->head_rounds = head / workers;
  plan->tail_items = n_tail;
  plan->tail_splits = 0;
  plan->n_units = head + pieces;
  plan->grid = workers * cpi;
  plan->kernels_per_call = split_items > 0 ? 2 : 1;
  plan->variant = variant;
  plan->total_tiles = total;
  plan->workspace_bytes =
      split_items > 0 ? 2 * static_cast<int64_t>(workers) * cpi * kRowsPerTile * kPartialRowBytes : 0;
  plan->est_makespan_tiles = *std::max_element(load.begin(), load.end());
  double us = static_cast<double>(plan->est_makespan_tiles) * (variant == 2 ? kPairTileUs : kTileUs);
  if (split_items > 0) {
    const double bytes = static_cast<double>(cpi * kRowsPerTile) *
                         (split_items * 520.0 + partial * static_cast<double>(kPartialRowBytes));
    us += bytes / kMergeBytesPerUs + kMergeLaunchUs;
  }
  return us;
}

// Best plan of one variant: searches the number of whole rounds (the last few
// full rounds and none) and the tail's cut (uniform S-way splits or the
// balanced tail); a split must win by 2 % over the simpler plan to be taken.
// force_splits: S > 0 forces the uniform cut with S pieces, kForceBalanced the
// balanced tail (the best number of whole rounds for it, if any fits).
double best_plan_of(const std::vector<SeqIn>& seqs, int num_sms, int variant, int workers,
                    int force_splits, gqa_prefill_plan* plan) {
  static thread_local Batch b;  // large: not on the stack
  build_batch(seqs, variant, &b);
  const std::vector<int> tiles = item_tile_counts(b);
  int q_tiles = 0;
  for (int i = 0; i < b.n_seq; ++i) q_tiles += b.seq[i].n_qtiles;
  const int n_items = static_cast<int>(tiles.size());
  const int max_splits = std::max(1, *std::min_element(tiles.begin(), tiles.end()));
  const int full_rounds = n_items / workers;
  if (force_splits > 0)
    return plan_schedule(tiles, q_tiles, num_sms, variant, workers, full_rounds,
                         std::min(force_splits, max_splits), plan);
  double best = plan_schedule(tiles, q_tiles, num_sms, variant, workers, 0, 1, plan);
  gqa_prefill_plan cand{};
  if (force_splits == kForceBalanced) {
    double best_b = -1.0;
    for (int hr = full_rounds; hr >= 0; --hr) {
      const double us = plan_balanced(tiles, q_tiles, num_sms, variant, workers, hr, &cand);
      if (us >= 0.0 && (best_b < 0.0 || us < best_b)) {
        best_b = us;
        *plan = cand;
      }
    }
    return best_b >= 0.0 ? best_b : best;
  }
  for (int hr = full_rounds; hr >= 0; --hr) {
    if (hr < full_rounds - 3 && hr != 0) continue;
    for (int S : kSplitCandidates) {
      if (S == 1 || S > max_splits) continue;
      const double us = plan_schedule(tiles, q_tiles, num_sms, variant, workers, hr, S, &cand);
      if (us < 0.98 * best) {
        best = us;
        *plan = cand;
      }
    }
  }
  return best;
}

// Pure function of its arguments (seqs: at least one non-empty sequence).
// max_pairs: CTA pairs that can be resident at once. force_grid caps the CTAs
// launched (a pair counts as two).
void compute_plan(const std::vector<SeqIn>& seqs, int num_sms, int max_pairs, int force_splits,
                  int force_grid, int force_variant, bool paged, gqa_prefill_plan* plan) {
  const int cap = force_grid > 0 ? std::min(force_grid, num_sms) : num_sms;
  const int workers1 = std::max(1, cap);
  const int workers2 = std::max(1, std::min(max_pairs, cap / 2));
  if (force_variant == 1 || (force_variant == 0 && max_pairs < 1)) {
    best_plan_of(seqs, num_sms, 1, workers1, force_splits, plan);
    return;
  }
  if (force_variant == 2) {
    best_plan_of(seqs, num_sms, 2, workers2, force_splits, plan);
    return;
  }
  gqa_prefill_plan one{}, pair{};
  const double t1 = best_plan_of(seqs, num_sms, 1, workers1, force_splits, &one) *
                    (paged ? kPagedOneCtaFactor : 1.0);
  const double t2 = best_plan_of(seqs, num_sms, 2, workers2, force_splits, &pair);
  *plan = t2 < 0.98 * t1 ? pair : one;
}

// Plans keyed by everything they depend on: the device, the options, dense or
// paged K/V and the (q_len, kv_len) of every sequence in the caller's order.
void cached_plan(const std::vector<SeqIn>& seqs, int num_sms, int max_pairs, int force_splits,
                 int force_grid, int force_variant, bool paged, gqa_prefill_plan* plan) {
  static std::mutex mu;
  static std::map<std::vector<int>, gqa_prefill_plan> cache;
  std::vector<int> key{num_sms, max_pairs, force_splits, force_grid, force_variant, paged ? 1 : 0};
  for (const SeqIn& s : seqs) {
    key.push_back(s.q_len);
    key.push_back(s.kv_len);
  }
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      *plan = it->second;
      return;
    }
  }
  compute_plan(seqs, num_sms, max_pairs, force_splits, force_grid, force_variant, paged, plan);
  std::lock_guard<std::mutex> lock(mu);
  if (cache.size() > 4096) cache.clear();
  cache.emplace(std::move(key), *plan);
}

// --------------------------------------------------------------- validation --

bool misaligned(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0; }

gqa_status validate_heads(int n_q_heads, int n_kv_heads, int head_dim, float scale) {
  if (!(std::isfinite(scale) && scale > 0.0f)) return GQA_ERR_SHAPE;
  if (n_q_heads != kQHeads || n_kv_heads != kKvHeads || head_dim != kHeadDim)
    return GQA_ERR_UNSUPPORTED;
  return GQA_OK;
}

// Sequences of a batched call from the caller's HOST arrays: query rows
// cu_q[b] .. cu_q[b+1]-1 and, with dense K/V, key rows cu_k[b] .. cu_k[b+1]-1;
// with paged K/V (cu_k null) kv_lens[b] keys through block-table row b.
gqa_status batch_from_host(const int32_t* cu_q, const int32_t* cu_k, const int32_t* kv_lens,
                           int batch, std::vector<SeqIn>* seqs, int* total_q, int64_t* total_kv) {
  if (batch < 0) return GQA_ERR_SHAPE;
  if (batch > kMaxSeqs) return GQA_ERR_UNSUPPORTED;
  seqs->clear();
  *total_q = 0;
  *total_kv = 0;
  if (batch == 0) return GQA_OK;
  if (!cu_q || (!cu_k && !kv_lens)) return GQA_ERR_NULL;
  if (cu_q[0] != 0 || (cu_k && cu_k[0] != 0)) return GQA_ERR_SHAPE;
  for (int b = 0; b < batch; ++b) {
    const int q_len = cu_q[b + 1] - cu_q[b];
    const int kv_len = cu_k ? cu_k[b + 1] - cu_k[b] : kv_lens[b];
    if (cu_q[b + 1] < cu_q[b] || kv_len < 0 || q_len > kv_len) return GQA_ERR_SHAPE;
    seqs->push_back(SeqIn{cu_q[b], q_len, cu_k ? cu_k[b] : 0, kv_len, 0});
  }
  *total_q = cu_q[batch];
  *total_kv = cu_k ? cu_k[batch] : 0;
  return GQA_OK;
}

// ------------------------------------------------------------ device state --
// Per-device facts both entry points need: SM count, co-resident CTA pairs and
// the status word's device address. Set up once per device with it current; no
// device memory is allocated here.
struct DeviceInfo {
  std::once_flag once;
  gqa_status status = GQA_OK;
  int num_sms = 0;
  int max_pairs = 0;
  int* status_word = nullptr;
};
DeviceInfo g_info[kMaxDevices];

gqa_status device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GQA_ERR_CUDA;
  DeviceInfo& s = g_info[dev];
  std::call_once(s.once, [&s, dev] {
    cudaDeviceProp prop{};
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) { s.status = GQA_ERR_CUDA; return; }
    // The kernels are built for sm_103a only (tcgen05 / TMEM / TMA).
    if (!(prop.major == 10 && prop.minor == 3)) { s.status = GQA_ERR_UNSUPPORTED; return; }
    s.num_sms = prop.multiProcessorCount;
    if (prepare_fwd_kernel() != cudaSuccess || status_word_address(&s.status_word) != cudaSuccess) {
      s.status = GQA_ERR_CUDA;
      return;
    }
    int pairs = 0;
    if (max_active_pairs(&pairs) != cudaSuccess) pairs = 0;  // then the pair kernel is not used
    s.max_pairs = std::min(pairs, s.num_sms / 2);
  });
  if (s.status != GQA_OK) return s.status;
  *out = &s;
  return GQA_OK;
}

// The stream-ordered pool that gqa_prefill_attn takes split partials from.
struct DevicePool {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  cudaMemPool_t pool = nullptr;
};
DevicePool g_pool[kMaxDevices];

gqa_status device_pool(cudaMemPool_t* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GQA_ERR_CUDA;
  DevicePool& s = g_pool[dev];
  std::call_once(s.once, [&s, dev] {
    cudaMemPoolProps props{};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    if ((s.err = cudaMemPoolCreate(&s.pool, &props)) != cudaSuccess) return;
    uint64_t keep = UINT64_MAX;  // keep freed partial buffers cached in the pool
    s.err = cudaMemPoolSetAttribute(s.pool, cudaMemPoolAttrReleaseThreshold, &keep);
  });
  if (s.err != cudaSuccess) return GQA_ERR_CUDA;
  *out = s.pool;
  return GQA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// One tiled tensor map; dims/strides/box as cuTensorMapEncodeTiled takes them
// (strides in bytes for dims 1..rank-1), unit element strides.
bool encode(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
            const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
            CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(map, dtype, static_cast<cuuint32_t>(rank), const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Element type of the Q and K tensors: BF16 values, or E4M3 codes (one byte).
struct Elem {
  CUtensorMapDataType dtype;
  uint32_t bytes;
};
constexpr Elem kBf16{CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2};
constexpr Elem kE4m3{CU_TENSOR_MAP_DATA_TYPE_UINT8, 1};

// Q [q_len][24][256]: box (one 128-byte chunk of d, 6 heads, 21 tokens).
bool encode_q(CUtensorMap* map, const void* base, uint64_t q_len, Elem e) {
  const cuuint64_t dims[3] = {kHeadDim, kQHeads, q_len};
  const cuuint64_t strides[2] = {kHeadDim * e.bytes, static_cast<cuuint64_t>(kQHeads) * kHeadDim * e.bytes};
  const cuuint32_t box[3] = {128 / e.bytes, static_cast<cuuint32_t>(kGroup), kTokPerTile};
  return encode(map, e.dtype, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// K or V [rows][4 heads][256] as a 4-D tensor (one 128-byte chunk of d, row,
// head, chunk) with the chunk outermost, so that one box of (chunk, box_rows,
// 1, box_chunks) lands in shared memory chunk-major: chunk c's box_rows rows of
// 128 bytes at c * box_rows * 128, as the MMA descriptors read them.
bool encode_kv(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows,
               uint32_t box_chunks, Elem e) {
  const cuuint64_t per_chunk = 128 / e.bytes;
  const cuuint64_t dims[4] = {per_chunk, rows, static_cast<cuuint64_t>(kKvHeads),
                              kHeadDim / per_chunk};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(kKvHeads) * kHeadDim * e.bytes,  // key
                                 kHeadDim * e.bytes,                                       // head
                                 128};                                                     // chunk
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(per_chunk), box_rows, 1, box_chunks};
  return encode(map, e.dtype, 4, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// A paged K or V cache [rows][4 heads][256] (rows a multiple of 16; BF16 values
// or E4M3 codes) as a 5-D tensor (one 128-byte chunk of d, key % 8, chunk,
// key / 8, head): one box of (chunk, 8, box_chunks, box_rows / 8, 1) lands in
// shared memory as 8-key groups, each holding its box_chunks chunks of 8 rows x
// 128 bytes — the paged stage layout of the attention kernel, in which a piece
// of whole 8-key groups is contiguous.
bool encode_kv_paged(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows,
                     uint32_t box_chunks, Elem e = kBf16) {
  const cuuint64_t per_chunk = 128 / e.bytes;
  const cuuint64_t row_bytes = static_cast<cuuint64_t>(kKvHeads) * kHeadDim * e.bytes;
  const cuuint64_t dims[5] = {per_chunk, 8, kHeadDim / per_chunk, rows / 8,
                              static_cast<cuuint64_t>(kKvHeads)};
  const cuuint64_t strides[4] = {row_bytes,            // next key in the group
                                 128,                  // next chunk
                                 8 * row_bytes,        // next group of 8 keys
                                 kHeadDim * e.bytes};  // next head
  const cuuint32_t box[5] = {static_cast<cuuint32_t>(per_chunk), 8, box_chunks, box_rows / 8, 1};
  return encode(map, e.dtype, 5, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Key scales FP32 [4 heads][stride], box (128 keys, 1 head); keys past kv_len
// read zeros.
bool encode_key_scales(CUtensorMap* map, const float* base, uint64_t kv_len, uint64_t stride) {
  const cuuint64_t dims[2] = {kv_len, static_cast<cuuint64_t>(kKvHeads)};
  const cuuint64_t strides[1] = {stride * 4};
  const cuuint32_t box[2] = {kBlockN, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box,
                CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Pointers of a call that has work to do (with none, they may be NULL).
gqa_status check_pointers(const void* q, const void* k, const void* v, const void* out,
                          const float* lse) {
  if (!q || !k || !v || !out) return GQA_ERR_NULL;
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(out) || misaligned(lse))
    return GQA_ERR_ALIGN;
  return GQA_OK;
}

// K/V of a paged call: the caches span num_pages * page_size rows; sequence
// b's block-table row starts at b * bt_stride.
struct PagedKV {
  const int32_t* block_table;
  int bt_stride;
  int num_pages;
  int page_size;
};
constexpr int64_t kMaxCacheRows = int64_t{1} << 30;  // TMA row coordinates stay far from 2^31

gqa_status check_paged(const PagedKV& pkv, const std::vector<SeqIn>& seqs, bool work) {
  if (pkv.page_size <= 0 || pkv.page_size % 16 != 0) return GQA_ERR_UNSUPPORTED;
  if (pkv.num_pages < 1 || static_cast<int64_t>(pkv.num_pages) * pkv.page_size >= kMaxCacheRows)
    return GQA_ERR_SHAPE;
  for (const SeqIn& s : seqs)  // every row must hold the sequence's pages
    if (seqs.size() > 1 && (s.kv_len + pkv.page_size - 1) / pkv.page_size > pkv.bt_stride)
      return GQA_ERR_SHAPE;
  if (!work) return GQA_OK;
  if (!pkv.block_table) return GQA_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(pkv.block_table) & 3u) != 0) return GQA_ERR_ALIGN;
  return GQA_OK;
}

// Quantised-QK^T inputs of a call: q and k are E4M3 codes with these scales;
// with v_scale set, v is also E4M3 codes, transposed ([4][256][v_stride]).
struct Fp8Qk {
  const float* q_scale;  // [q_len][24]
  const float* k_scale;  // [4][k_scale_stride]
  int k_scale_stride;
  const float* v_scale = nullptr;  // [4][256] per-channel scales (quantised PV)
  int v_stride = 0;                // bytes between channel rows of the V codes
};

// V codes of the quantised PV, [4 heads][256 channels][v_stride keys] bytes, as a
// 3-D tensor (key, channel, head) of kv_len keys (keys past it read zeros); box
// (128 keys, box_ch channels, 1 head) lands as box_ch rows of 128 bytes (K-major).
bool encode_v_codes(CUtensorMap* map, const void* base, uint64_t kv_len, uint64_t v_stride,
                    uint32_t box_ch) {
  const cuuint64_t dims[3] = {kv_len, kHeadDim, static_cast<cuuint64_t>(kKvHeads)};
  const cuuint64_t strides[2] = {v_stride, v_stride * kHeadDim};
  const cuuint32_t box[3] = {kBlockN, box_ch, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box,
                CU_TENSOR_MAP_SWIZZLE_128B);
}

gqa_status check_fp8(const Fp8Qk& f8, int64_t key_rows, bool work, bool pv) {
  if (f8.k_scale_stride < key_rows || f8.k_scale_stride % 4 != 0 ||
      static_cast<int64_t>(f8.k_scale_stride) * kKvHeads >= (int64_t{1} << 31))
    return GQA_ERR_SHAPE;
  if (pv && (f8.v_stride < key_rows || f8.v_stride % 16 != 0 ||
             static_cast<int64_t>(f8.v_stride) * kHeadDim * kKvHeads >= (int64_t{1} << 40)))
    return GQA_ERR_SHAPE;
  if (!work) return GQA_OK;
  if (!f8.q_scale || !f8.k_scale || (pv && !f8.v_scale)) return GQA_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(f8.q_scale) & 3u) != 0 || misaligned(f8.k_scale) ||
      (pv && misaligned(f8.v_scale)))
    return GQA_ERR_ALIGN;
  return GQA_OK;
}

int gcd_int(int a, int b) {
  while (b != 0) {
    const int t = a % b;
    a = b;
    b = t;
  }
  return a;
}

// Tensors and options of one call.
struct CallIO {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  float* lse;
  const PagedKV* pkv;  // null: dense K/V; else k and v are the paged caches
  const Fp8Qk* f8;     // null: BF16 Q/K; else q and k are E4M3 codes with these scales
  float scale;
};

// Launches `plan` on `stream`; `ws` holds plan.workspace_bytes (or nothing).
// total_q / total_kv: rows of the packed Q and (dense) K/V.
gqa_status launch_plan(const gqa_prefill_plan& plan, const CallIO& io,
                       const std::vector<SeqIn>& seqs, int total_q, int64_t total_kv,
                       int* status_word, void* ws, const gqa_prefill_opts* opts,
                       cudaStream_t stream) {
  const bool pair = plan.variant == 2;
  static thread_local FwdParams p;  // ~5 KB with the sequence table: not on the stack
  std::memset(&p, 0, sizeof(p));
  const uint64_t kv_rows = io.pkv ? static_cast<uint64_t>(io.pkv->num_pages) * io.pkv->page_size
                                  : static_cast<uint64_t>(total_kv);
  const Elem qk = io.f8 ? kE4m3 : kBf16;
  // K/V stages per CTA: one-CTA K 128 keys (BF16: 2 chunks per stage, 2 stages;
  // FP8: all 2 chunks), V 64 keys x 4 chunks; pairs K 64 keys x all chunks,
  // V 128 keys x 2 chunks.
  const uint32_t k_rows = pair ? 64 : kBlockN;
  const uint32_t k_chunks = io.f8 ? 2 : (pair ? 4 : 2);
  const uint32_t v_rows = pair ? kBlockN : 64, v_chunks = pair ? 2 : 4;
  const bool fp8_pv = io.f8 && io.f8->v_scale;
  if (!encode_q(&p.tmap_q, io.q, static_cast<uint64_t>(total_q), qk)) return GQA_ERR_CUDA;
  if (!io.pkv) {
    if (!encode_kv(&p.tmap_k, io.k, kv_rows, k_rows, k_chunks, qk) ||
        !(fp8_pv ? encode_v_codes(&p.tmap_v, io.v, kv_rows,
                                  static_cast<uint64_t>(io.f8->v_stride), pair ? 128 : 256)
                 : encode_kv(&p.tmap_v, io.v, kv_rows, v_rows, v_chunks, kBf16)))
      return GQA_ERR_CUDA;
    if (seqs.size() > 1) {
      // A box past a sequence's last key would read the next sequence's values:
      // that tile's V goes in 16-key pieces (see the kernel's issue_dense_v_pieces).
      if (!encode_kv(&p.tmap_v16, io.v, kv_rows, 16, 1, kBf16)) return GQA_ERR_CUDA;
      p.oob_row = static_cast<int>(kv_rows);
    }
  } else {
    const PagedKV& pkv = *io.pkv;
    const uint32_t sub = static_cast<uint32_t>(gcd_int(pkv.page_size, 64));  // 16, 32 or 64
    if (!encode_kv_paged(&p.tmap_k, io.k, kv_rows, k_rows, k_chunks, qk) ||
        !encode_kv_paged(&p.tmap_v, io.v, kv_rows, v_rows, v_chunks) ||
        !encode_kv_paged(&p.tmap_k_sub, io.k, kv_rows, sub, k_chunks, qk) ||
        !encode_kv_paged(&p.tmap_v_sub, io.v, kv_rows, sub, v_chunks) ||
        !encode_kv_paged(&p.tmap_v16, io.v, kv_rows, 16, v_chunks))
      return GQA_ERR_CUDA;
    p.block_table = pkv.block_table;
    p.bt_stride = pkv.bt_stride;
    p.page_size = pkv.page_size;
    p.num_pages = pkv.num_pages;
    p.sub_rows = static_cast<int>(sub);
    p.oob_row = static_cast<int>(kv_rows);
  }
  if (io.f8) {
    // One scale per key row of K: the packed keys (each sequence from a column that
    // is a multiple of 4), or every row of the paged cache.
    uint64_t scale_rows = kv_rows;
    if (!io.pkv) {
      scale_rows = 0;
      for (const SeqIn& sq : seqs) {
        if (sq.ks_start % 4 != 0) return GQA_ERR_ALIGN;  // every TMA start on 16 bytes
        scale_rows = std::max<uint64_t>(scale_rows, static_cast<uint64_t>(sq.ks_start) + sq.kv_len);
      }
    }
    const uint64_t stride = static_cast<uint64_t>(io.f8->k_scale_stride);
    if (!io.pkv && !encode_key_scales(&p.tmap_ks, io.f8->k_scale, scale_rows, stride))
      return GQA_ERR_CUDA;
    p.k_scale = io.f8->k_scale;
    p.k_scale_stride = io.f8->k_scale_stride;
    p.q_scale = io.f8->q_scale;
    p.v_scale = io.f8->v_scale;
  }
  build_batch(seqs, plan.variant, &p.batch);
  const int workers = pair ? plan.grid / 2 : plan.grid;
  p.out = static_cast<__nv_bfloat16*>(io.out);
  p.lse = io.lse;
  p.status = status_word;
  p.out_rows = static_cast<long long>(total_q) * kQHeads;
  p.part_rows = 0;
  p.head_items = std::min(plan.head_rounds * workers, plan.n_items);
  p.tail_splits = plan.tail_splits;
  p.n_units = plan.n_units;
  p.n_tail = 0;
  if (plan.tail_splits == 0) {  // balanced tail: tile prefix sums of the tail items
    p.n_tail = plan.n_items - p.head_items;
    p.tail.v[0] = 0;
    for (int k = 0; k < p.n_tail; ++k) {
      int seq, qt, g;
      item_of(p.batch, p.head_items + k, seq, qt, g);
      p.tail.v[k + 1] = p.tail.v[k] + item_tiles(p.batch.seq[seq], p.batch.tok_per_item, qt);
    }
  }
  p.scale_log2 = io.scale * 1.4426950408889634f;
  p.timeout_ns = (opts && opts->wait_timeout_us) ? 1000ull * opts->wait_timeout_us
                                                 : kDefaultTimeoutNs;
  p.withhold_q = (opts && opts->test_withhold_q) ? 1 : 0;
  // Every chunk within one query tile of an item: each KV tile of a sequence and
  // group belongs to exactly one item, so no tile is read twice.
  p.kv_read_once = 1;
  for (const SeqIn& sq : seqs)
    if (sq.q_len > p.batch.tok_per_item) p.kv_read_once = 0;
  if (plan.workspace_bytes > 0) {
    // Partial slots: tail_items * S (uniform tail) or two per worker (balanced).
    const size_t slots = plan.tail_splits > 0
                             ? static_cast<size_t>(plan.tail_items) * plan.tail_splits
                             : 2 * static_cast<size_t>(workers);
    p.part_o = static_cast<float*>(ws);
    p.part_lse = p.part_o + slots * (pair ? 2 : 1) * kRowsPerTile * kHeadDim;
    p.part_rows = static_cast<long long>(slots) * (pair ? 2 : 1) * kRowsPerTile;
  }
  auto ev_begin = static_cast<cudaEvent_t>(opts ? opts->fwd_event_begin : nullptr);
  auto ev_end = static_cast<cudaEvent_t>(opts ? opts->fwd_event_end : nullptr);
  if (ev_begin && cudaEventRecord(ev_begin, stream) != cudaSuccess) return GQA_ERR_CUDA;
  const int kv_mode = io.pkv ? 1 : (seqs.size() > 1 ? 2 : 0);
  if (launch_fwd(p, plan.grid, pair, kv_mode, io.f8 ? (fp8_pv ? 2 : 1) : 0, stream) != cudaSuccess)
    return GQA_ERR_CUDA;
  if (ev_end && cudaEventRecord(ev_end, stream) != cudaSuccess) return GQA_ERR_CUDA;
  if (plan.kernels_per_call == 2) {  // the separate merge pass
    static thread_local MergeParams m;
    m.part_o = p.part_o;
    m.part_lse = p.part_lse;
    m.out = p.out;
    m.lse = io.lse;
    m.status = p.status;
    m.out_rows = p.out_rows;
    m.part_rows = p.part_rows;
    m.head_items = p.head_items;
    m.tail_items = plan.tail_items;
    m.tail_splits = plan.tail_splits;
    m.workers = workers;
    m.ctas_per_item = pair ? 2 : 1;
    m.tail = p.tail;
    m.batch = p.batch;
    if (launch_merge(m, stream) != cudaSuccess) return GQA_ERR_CUDA;
  }
  return GQA_OK;
}

// Every entry point but the allocation-free one: check, plan, take split
// partials from the pool, launch.
gqa_status run(const CallIO& io, const std::vector<SeqIn>& seqs, int total_q, int64_t total_kv,
               int n_q_heads, int n_kv_heads, int head_dim, void* stream_ptr,
               const gqa_prefill_opts* opts, gqa_prefill_plan* plan_out) {
  if (plan_out) std::memset(plan_out, 0, sizeof(*plan_out));
  gqa_status st = validate_heads(n_q_heads, n_kv_heads, head_dim, io.scale);
  const bool work = total_q > 0;
  if (st == GQA_OK && work) st = check_pointers(io.q, io.k, io.v, io.out, io.lse);
  if (st == GQA_OK && work && io.f8 && io.f8->v_scale && io.f8->v_stride % 16 != 0)
    st = GQA_ERR_SHAPE;
  if (st == GQA_OK && io.pkv) st = check_paged(*io.pkv, seqs, work);
  if (st == GQA_OK && io.f8) {
    int64_t scale_cols = static_cast<int64_t>(io.pkv ? io.pkv->num_pages : 0) *
                         (io.pkv ? io.pkv->page_size : 0);
    if (!io.pkv) {  // dense: every sequence's scales start on a multiple of 4
      std::vector<SeqIn> tmp = seqs;
      scale_cols = key_scale_starts(&tmp);
    }
    st = check_fp8(*io.f8, scale_cols, work, io.f8->v_scale != nullptr);
    // Quantised PV: one sequence, dense K/V (V's channel scales span the call's keys).
    if (st == GQA_OK && io.f8->v_scale && (io.pkv || seqs.size() != 1)) st = GQA_ERR_UNSUPPORTED;
  }
  if (st != GQA_OK || !work) return st;
  std::vector<SeqIn> fp8_seqs;
  const std::vector<SeqIn>* use = &seqs;
  if (io.f8 && !io.pkv) {
    fp8_seqs = seqs;
    key_scale_starts(&fp8_seqs);
    use = &fp8_seqs;
  }
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != GQA_OK) return st;
  gqa_prefill_plan plan{};
  cached_plan(seqs, dev->num_sms, dev->max_pairs, opts ? opts->force_splits : 0,
              opts ? opts->force_grid : 0, opts ? opts->force_variant : 0, io.pkv != nullptr,
              &plan);
  if (plan_out) *plan_out = plan;
  auto stream = static_cast<cudaStream_t>(stream_ptr);
  void* ws = nullptr;
  if (plan.workspace_bytes > 0) {
    cudaMemPool_t pool = nullptr;
    if ((st = device_pool(&pool)) != GQA_OK) return st;
    if (cudaMallocFromPoolAsync(&ws, static_cast<size_t>(plan.workspace_bytes), pool, stream) !=
        cudaSuccess)
      return GQA_ERR_CUDA;
  }
  st = launch_plan(plan, io, *use, total_q, total_kv, dev->status_word, ws, opts, stream);
  if (ws && cudaFreeAsync(ws, stream) != cudaSuccess) st = GQA_ERR_CUDA;
  return st;
}

// One sequence: q_len tokens at the end of kv_len keys (the non-batched calls).
gqa_status run_one(const CallIO& io, int q_len, int kv_len, int n_q_heads, int n_kv_heads,
                   int head_dim, void* stream, const gqa_prefill_opts* opts,
                   gqa_prefill_plan* plan_out) {
  if (plan_out) std::memset(plan_out, 0, sizeof(*plan_out));
  if (q_len < 0 || kv_len < q_len) return GQA_ERR_SHAPE;
  const std::vector<SeqIn> seqs{SeqIn{0, q_len, 0, kv_len, 0}};
  return run(io, seqs, q_len, kv_len, n_q_heads, n_kv_heads, head_dim, stream, opts, plan_out);
}

// ---------------------------------------------------- allocation-free variant --
// Split-KV partials of gqa_prefill_attn_noalloc live in this file-scope array
// instead of the stream-ordered pool. In host code `g_noalloc_scratch` is only a
// host-side stand-in for the symbol: its device address comes from
// cudaGetSymbolAddress, once per device, with that device current.
constexpr size_t kNoAllocScratchBytes = GQA_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The lookup is retried until it succeeds: a failed first attempt (say, one made
// while the stream was being captured) does not disable the entry point.
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};  // device address of g_noalloc_scratch per device

gqa_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GQA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_addr[dev] == nullptr) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_noalloc_scratch) != cudaSuccess || a == nullptr) {
      cudaGetLastError();  // do not leave the failure for the caller's next CUDA call
      return GQA_ERR_CUDA;
    }
    g_noalloc_addr[dev] = a;
  }
  *out = g_noalloc_addr[dev];
  return GQA_OK;
}

gqa_status run_noalloc(const void* q, const void* k, const void* v, void* out, float* lse,
                       int q_len, int kv_len, int n_q_heads, int n_kv_heads, int head_dim,
                       float scale, void* stream_ptr) {
  if (q_len < 0 || kv_len < q_len) return GQA_ERR_SHAPE;
  gqa_status st = validate_heads(n_q_heads, n_kv_heads, head_dim, scale);
  if (st != GQA_OK || q_len == 0) return st;
  if ((st = check_pointers(q, k, v, out, lse)) != GQA_OK) return st;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != GQA_OK) return st;
  void* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != GQA_OK) return st;
  const std::vector<SeqIn> seqs{SeqIn{0, q_len, 0, kv_len, 0}};
  gqa_prefill_plan plan{};
  cached_plan(seqs, dev->num_sms, dev->max_pairs, 0, 0, 0, false, &plan);
  if (static_cast<uint64_t>(plan.workspace_bytes) > kNoAllocScratchBytes) return GQA_ERR_SCRATCH;
  // Every partial row the merge reads is written by the attention kernel first,
  // so the scratch needs no clearing between calls.
  const CallIO io{q, k, v, out, lse, nullptr, nullptr, scale};
  return launch_plan(plan, io, seqs, q_len, kv_len, dev->status_word, scratch, nullptr,
                     static_cast<cudaStream_t>(stream_ptr));
}

}  // namespace
}  // namespace gqa

extern "C" {

gqa_status gqa_prefill_attn_noalloc(const void* q, const void* k, const void* v, void* out,
                                    float* lse, int q_len, int kv_len, int n_q_heads,
                                    int n_kv_heads, int head_dim, float scale, void* stream) {
  return gqa::run_noalloc(q, k, v, out, lse, q_len, kv_len, n_q_heads, n_kv_heads, head_dim,
                          scale, stream);
}


gqa_status gqa_prefill_attn(const void* q, const void* k, const void* v, void* out, float* lse,
                            int q_len, int kv_len, int n_q_heads, int n_kv_heads, int head_dim,
                            float scale, void* stream) {
  const gqa::CallIO io{q, k, v, out, lse, nullptr, nullptr, scale};
  return gqa::run_one(io, q_len, kv_len, n_q_heads, n_kv_heads, head_dim, stream, nullptr,
                      nullptr);
}

gqa_status gqa_prefill_attn_ex(const void* q, const void* k, const void* v, void* out, float* lse,
                               int q_len, int kv_len, int n_q_heads, int n_kv_heads, int head_dim,
                               float scale, void* stream, const gqa_prefill_opts* opts,
                               gqa_prefill_plan* plan_out) {
  const gqa::CallIO io{q, k, v, out, lse, nullptr, nullptr, scale};
  return gqa::run_one(io, q_len, kv_len, n_q_heads, n_kv_heads, head_dim, stream, opts, plan_out);
}

gqa_status gqa_prefill_attn_paged(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_table, int num_pages, int page_size,
                                  void* out, float* lse, int q_len, int kv_len, int n_q_heads,
                                  int n_kv_heads, int head_dim, float scale, void* stream) {
  return gqa_prefill_attn_paged_ex(q, k_cache, v_cache, block_table, num_pages, page_size, out,
                                   lse, q_len, kv_len, n_q_heads, n_kv_heads, head_dim, scale,
                                   stream, nullptr, nullptr);
}

gqa_status gqa_prefill_attn_paged_ex(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_table, int num_pages, int page_size,
                                     void* out, float* lse, int q_len, int kv_len,
                                     int n_q_heads, int n_kv_heads, int head_dim, float scale,
                                     void* stream, const gqa_prefill_opts* opts,
                                     gqa_prefill_plan* plan_out) {
  const gqa::PagedKV pkv{block_table, 0, num_pages, page_size};
  const gqa::CallIO io{q, k_cache, v_cache, out, lse, &pkv, nullptr, scale};
  return gqa::run_one(io, q_len, kv_len, n_q_heads, n_kv_heads, head_dim, stream, opts, plan_out);
}

gqa_status gqa_prefill_attn_varlen_ex(const void* q, const void* k, const void* v, void* out,
                                      float* lse, const int32_t* cu_seqlens_q,
                                      const int32_t* cu_seqlens_k, int batch, int n_q_heads,
                                      int n_kv_heads, int head_dim, float scale, void* stream,
                                      const gqa_prefill_opts* opts, gqa_prefill_plan* plan_out) {
  if (plan_out) std::memset(plan_out, 0, sizeof(*plan_out));
  if (batch > 0 && !cu_seqlens_k) return GQA_ERR_NULL;
  std::vector<gqa::SeqIn> seqs;
  int total_q = 0;
  int64_t total_kv = 0;
  const gqa_status st = gqa::batch_from_host(cu_seqlens_q, cu_seqlens_k, nullptr, batch, &seqs,
                                             &total_q, &total_kv);
  if (st != GQA_OK) return st;
  const gqa::CallIO io{q, k, v, out, lse, nullptr, nullptr, scale};
  return gqa::run(io, seqs, total_q, total_kv, n_q_heads, n_kv_heads, head_dim, stream, opts,
                  plan_out);
}

gqa_status gqa_prefill_attn_varlen(const void* q, const void* k, const void* v, void* out,
                                   float* lse, const int32_t* cu_seqlens_q,
                                   const int32_t* cu_seqlens_k, int batch, int n_q_heads,
                                   int n_kv_heads, int head_dim, float scale, void* stream) {
  return gqa_prefill_attn_varlen_ex(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, batch,
                                    n_q_heads, n_kv_heads, head_dim, scale, stream, nullptr,
                                    nullptr);
}

gqa_status gqa_prefill_attn_paged_varlen_ex(const void* q, const void* k_cache,
                                            const void* v_cache, const int32_t* block_table,
                                            int bt_stride, int num_pages, int page_size,
                                            void* out, float* lse,
                                            const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                                            int batch, int n_q_heads, int n_kv_heads,
                                            int head_dim, float scale, void* stream,
                                            const gqa_prefill_opts* opts,
                                            gqa_prefill_plan* plan_out) {
  if (plan_out) std::memset(plan_out, 0, sizeof(*plan_out));
  if (batch > 0 && !kv_lens) return GQA_ERR_NULL;
  if (bt_stride < 0) return GQA_ERR_SHAPE;
  std::vector<gqa::SeqIn> seqs;
  int total_q = 0;
  int64_t total_kv = 0;
  const gqa_status st =
      gqa::batch_from_host(cu_seqlens_q, nullptr, kv_lens, batch, &seqs, &total_q, &total_kv);
  if (st != GQA_OK) return st;
  const gqa::PagedKV pkv{block_table, bt_stride, num_pages, page_size};
  const gqa::CallIO io{q, k_cache, v_cache, out, lse, &pkv, nullptr, scale};
  return gqa::run(io, seqs, total_q, 0, n_q_heads, n_kv_heads, head_dim, stream, opts, plan_out);
}

gqa_status gqa_prefill_attn_paged_varlen(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_table, int bt_stride, int num_pages,
                                         int page_size, void* out, float* lse,
                                         const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                                         int batch, int n_q_heads, int n_kv_heads, int head_dim,
                                         float scale, void* stream) {
  return gqa_prefill_attn_paged_varlen_ex(q, k_cache, v_cache, block_table, bt_stride, num_pages,
                                          page_size, out, lse, cu_seqlens_q, kv_lens, batch,
                                          n_q_heads, n_kv_heads, head_dim, scale, stream, nullptr,
                                          nullptr);
}

namespace {
gqa::ScaleColumns one_sequence() {
  gqa::ScaleColumns c;
  std::memset(&c, 0, sizeof(c));
  c.n_seq = 1;
  return c;
}
}  // namespace

gqa_status gqa_quantize_q_fp8(const void* q, void* q_fp8, float* q_scale, int q_len,
                              int n_q_heads, int head_dim, void* stream) {
  if (q_len < 0) return GQA_ERR_SHAPE;
  if (n_q_heads != gqa::kQHeads || head_dim != gqa::kHeadDim) return GQA_ERR_UNSUPPORTED;
  if (q_len == 0) return GQA_OK;
  if (!q || !q_fp8 || !q_scale) return GQA_ERR_NULL;
  if (gqa::misaligned(q) || gqa::misaligned(q_fp8) || (reinterpret_cast<uintptr_t>(q_scale) & 3u))
    return GQA_ERR_ALIGN;
  gqa::DeviceInfo* di = nullptr;
  if (const gqa_status st = gqa::device_info(&di); st != GQA_OK) return st;
  return gqa::launch_quantize_fp8(q, q_fp8, q_scale, q_len, gqa::kQHeads, 0, false,
                                  one_sequence(), di->num_sms,
                                  static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? GQA_OK
             : GQA_ERR_CUDA;
}

gqa_status gqa_quantize_k_fp8(const void* k, void* k_fp8, float* k_scale, int kv_len,
                              int n_kv_heads, int head_dim, int k_scale_stride, void* stream) {
  if (kv_len < 0 || k_scale_stride < kv_len || k_scale_stride % 4 != 0 ||
      static_cast<int64_t>(k_scale_stride) * gqa::kKvHeads >= (int64_t{1} << 31))
    return GQA_ERR_SHAPE;
  if (n_kv_heads != gqa::kKvHeads || head_dim != gqa::kHeadDim) return GQA_ERR_UNSUPPORTED;
  if (kv_len == 0) return GQA_OK;
  if (!k || !k_fp8 || !k_scale) return GQA_ERR_NULL;
  if (gqa::misaligned(k) || gqa::misaligned(k_fp8) || gqa::misaligned(k_scale)) return GQA_ERR_ALIGN;
  gqa::DeviceInfo* di = nullptr;
  if (const gqa_status st = gqa::device_info(&di); st != GQA_OK) return st;
  return gqa::launch_quantize_fp8(k, k_fp8, k_scale, kv_len, gqa::kKvHeads, k_scale_stride, true,
                                  one_sequence(), di->num_sms,
                                  static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? GQA_OK
             : GQA_ERR_CUDA;
}

gqa_status gqa_quantize_k_fp8_varlen(const void* k, void* k_fp8, float* k_scale,
                                     const int32_t* cu_seqlens_k, int batch, int n_kv_heads,
                                     int head_dim, int k_scale_stride, void* stream) {
  if (batch < 0) return GQA_ERR_SHAPE;
  if (batch > gqa::kMaxSeqs) return GQA_ERR_UNSUPPORTED;
  if (n_kv_heads != gqa::kKvHeads || head_dim != gqa::kHeadDim) return GQA_ERR_UNSUPPORTED;
  if (batch == 0) return GQA_OK;
  if (!cu_seqlens_k) return GQA_ERR_NULL;
  if (cu_seqlens_k[0] != 0) return GQA_ERR_SHAPE;
  static thread_local gqa::ScaleColumns cols;
  std::memset(&cols, 0, sizeof(cols));
  cols.n_seq = batch;
  int64_t col = 0;
  for (int b = 0; b < batch; ++b) {
    const int kv_len = cu_seqlens_k[b + 1] - cu_seqlens_k[b];
    if (kv_len < 0) return GQA_ERR_SHAPE;
    cols.row_begin[b] = cu_seqlens_k[b];
    cols.col_begin[b] = static_cast<int>(col);
    col += (static_cast<int64_t>(kv_len) + 3) / 4 * 4;  // as the attention kernel reads them
  }
  cols.row_begin[batch] = cu_seqlens_k[batch];
  const int rows = cu_seqlens_k[batch];
  if (k_scale_stride < col || k_scale_stride % 4 != 0 ||
      static_cast<int64_t>(k_scale_stride) * gqa::kKvHeads >= (int64_t{1} << 31))
    return GQA_ERR_SHAPE;
  if (rows == 0) return GQA_OK;
  if (!k || !k_fp8 || !k_scale) return GQA_ERR_NULL;
  if (gqa::misaligned(k) || gqa::misaligned(k_fp8) || gqa::misaligned(k_scale)) return GQA_ERR_ALIGN;
  gqa::DeviceInfo* di = nullptr;
  if (const gqa_status st = gqa::device_info(&di); st != GQA_OK) return st;
  return gqa::launch_quantize_fp8(k, k_fp8, k_scale, rows, gqa::kKvHeads, k_scale_stride, true, cols,
                                  di->num_sms, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? GQA_OK
             : GQA_ERR_CUDA;
}

gqa_status gqa_prefill_attn_fp8qk(const void* q_fp8, const float* q_scale, const void* k_fp8,
                                  const float* k_scale, int k_scale_stride, const void* v,
                                  void* out, float* lse, int q_len, int kv_len, int n_q_heads,
                                  int n_kv_heads, int head_dim, float scale, void* stream) {
  const gqa::Fp8Qk f8{q_scale, k_scale, k_scale_stride};
  const gqa::CallIO io{q_fp8, k_fp8, v, out, lse, nullptr, &f8, scale};
  return gqa::run_one(io, q_len, kv_len, n_q_heads, n_kv_heads, head_dim, stream, nullptr,
                      nullptr);
}

gqa_status gqa_prefill_attn_fp8qk_ex(const void* q_fp8, const float* q_scale, const void* k_fp8,
                                     const float* k_scale, int k_scale_stride, const void* v,
                                     void* out, float* lse, int q_len, int kv_len, int n_q_heads,
                                     int n_kv_heads, int head_dim, float scale, void* stream,
                                     const gqa_prefill_opts* opts, gqa_prefill_plan* plan_out) {
  const gqa::Fp8Qk f8{q_scale, k_scale, k_scale_stride};
  const gqa::CallIO io{q_fp8, k_fp8, v, out, lse, nullptr, &f8, scale};
  return gqa::run_one(io, q_len, kv_len, n_q_heads, n_kv_heads, head_dim, stream, opts, plan_out);
}

gqa_status gqa_prefill_attn_fp8qk_varlen_ex(const void* q_fp8, const float* q_scale,
                                            const void* k_fp8, const float* k_scale,
                                            int k_scale_stride, const void* v, void* out,
                                            float* lse, const int32_t* cu_seqlens_q,
                                            const int32_t* cu_seqlens_k, int batch, int n_q_heads,
                                            int n_kv_heads, int head_dim, float scale,
                                            void* stream, const gqa_prefill_opts* opts,
                                            gqa_prefill_plan* plan_out) {
  if (plan_out) std::memset(plan_out, 0, sizeof(*plan_out));
  if (batch > 0 && !cu_seqlens_k) return GQA_ERR_NULL;
  std::vector<gqa::SeqIn> seqs;
  int total_q = 0;
  int64_t total_kv = 0;
  const gqa_status st = gqa::batch_from_host(cu_seqlens_q, cu_seqlens_k, nullptr, batch, &seqs,
                                             &total_q, &total_kv);
  if (st != GQA_OK) return st;
  const gqa::Fp8Qk f8{q_scale, k_scale, k_scale_stride};
  const gqa::CallIO io{q_fp8, k_fp8, v, out, lse, nullptr, &f8, scale};
  return gqa::run(io, seqs, total_q, total_kv, n_q_heads, n_kv_heads, head_dim, stream, opts,
                  plan_out);
}

gqa_status gqa_prefill_attn_paged_fp8qk_varlen_ex(
    const void* q_fp8, const float* q_scale, const void* k_cache_fp8, const float* k_scale,
    int k_scale_stride, const void* v_cache, const int32_t* block_table, int bt_stride,
    int num_pages, int page_size, void* out, float* lse, const int32_t* cu_seqlens_q,
    const int32_t* kv_lens, int batch, int n_q_heads, int n_kv_heads, int head_dim, float scale,
    void* stream, const gqa_prefill_opts* opts, gqa_prefill_plan* plan_out) {
  if (plan_out) std::memset(plan_out, 0, sizeof(*plan_out));
  if (batch > 0 && !kv_lens) return GQA_ERR_NULL;
  if (bt_stride < 0) return GQA_ERR_SHAPE;
  std::vector<gqa::SeqIn> seqs;
  int total_q = 0;
  int64_t total_kv = 0;
  const gqa_status st =
      gqa::batch_from_host(cu_seqlens_q, nullptr, kv_lens, batch, &seqs, &total_q, &total_kv);
  if (st != GQA_OK) return st;
  const gqa::PagedKV pkv{block_table, bt_stride, num_pages, page_size};
  const gqa::Fp8Qk f8{q_scale, k_scale, k_scale_stride};
  const gqa::CallIO io{q_fp8, k_cache_fp8, v_cache, out, lse, &pkv, &f8, scale};
  return gqa::run(io, seqs, total_q, 0, n_q_heads, n_kv_heads, head_dim, stream, opts, plan_out);
}

gqa_status gqa_quantize_v_fp8(const void* v, void* v_fp8t, float* v_scale, int kv_len,
                              int n_kv_heads, int head_dim, int v_stride, void* stream) {
  if (kv_len < 0 || v_stride < kv_len || v_stride % 16 != 0 ||
      static_cast<int64_t>(v_stride) * gqa::kHeadDim * gqa::kKvHeads >= (int64_t{1} << 40))
    return GQA_ERR_SHAPE;
  if (n_kv_heads != gqa::kKvHeads || head_dim != gqa::kHeadDim) return GQA_ERR_UNSUPPORTED;
  if (kv_len == 0) return GQA_OK;
  if (!v || !v_fp8t || !v_scale) return GQA_ERR_NULL;
  if (gqa::misaligned(v) || gqa::misaligned(v_fp8t) || gqa::misaligned(v_scale)) return GQA_ERR_ALIGN;
  return gqa::launch_quantize_v_fp8(v, v_fp8t, v_scale, kv_len, v_stride,
                                    static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? GQA_OK
             : GQA_ERR_CUDA;
}

gqa_status gqa_prefill_attn_fp8qkpv_ex(const void* q_fp8, const float* q_scale, const void* k_fp8,
                                       const float* k_scale, int k_scale_stride,
                                       const void* v_fp8t, const float* v_scale, int v_stride,
                                       void* out, float* lse, int q_len, int kv_len,
                                       int n_q_heads, int n_kv_heads, int head_dim, float scale,
                                       void* stream, const gqa_prefill_opts* opts,
                                       gqa_prefill_plan* plan_out) {
  gqa::Fp8Qk f8{q_scale, k_scale, k_scale_stride};
  f8.v_scale = v_scale;
  f8.v_stride = v_stride;
  if (!v_scale && q_len > 0) {
    if (plan_out) std::memset(plan_out, 0, sizeof(*plan_out));
    return GQA_ERR_NULL;
  }
  const gqa::CallIO io{q_fp8, k_fp8, v_fp8t, out, lse, nullptr, &f8, scale};
  return gqa::run_one(io, q_len, kv_len, n_q_heads, n_kv_heads, head_dim, stream, opts, plan_out);
}

gqa_status gqa_prefill_attn_fp8qkpv(const void* q_fp8, const float* q_scale, const void* k_fp8,
                                    const float* k_scale, int k_scale_stride, const void* v_fp8t,
                                    const float* v_scale, int v_stride, void* out, float* lse,
                                    int q_len, int kv_len, int n_q_heads, int n_kv_heads,
                                    int head_dim, float scale, void* stream) {
  return gqa_prefill_attn_fp8qkpv_ex(q_fp8, q_scale, k_fp8, k_scale, k_scale_stride, v_fp8t,
                                     v_scale, v_stride, out, lse, q_len, kv_len, n_q_heads,
                                     n_kv_heads, head_dim, scale, stream, nullptr, nullptr);
}

gqa_status gqa_prefill_make_plan(int q_len, int kv_len, int n_q_heads, int n_kv_heads, int head_dim,
                                 int num_sms, int max_pairs, int force_splits, int force_grid,
                                 int force_variant, gqa_prefill_plan* plan) {
  if (!plan) return GQA_ERR_NULL;
  const int32_t cu_q[2] = {0, q_len}, cu_k[2] = {0, kv_len};
  if (q_len < 0 || kv_len < q_len) return GQA_ERR_SHAPE;
  return gqa_prefill_make_plan_varlen(cu_q, cu_k, 1, n_q_heads, n_kv_heads, head_dim, num_sms,
                                      max_pairs, force_splits, force_grid, force_variant, plan);
}

gqa_status gqa_prefill_device_info(int* num_sms, int* max_pairs) {
  gqa::DeviceInfo* dev = nullptr;
  const gqa_status st = gqa::device_info(&dev);
  if (st != GQA_OK) return st;
  if (num_sms) *num_sms = dev->num_sms;
  if (max_pairs) *max_pairs = dev->max_pairs;
  return GQA_OK;
}

namespace {
// Host-only planning of a batch given as (cu_seqlens_q, cu_seqlens_k) (dense) or
// (cu_seqlens_q, kv_lens) (paged): the plan the attention call computes.
gqa_status host_plan(const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                     const int32_t* kv_lens, int batch, int n_q_heads, int n_kv_heads,
                     int head_dim, int num_sms, int max_pairs, int force_splits, int force_grid,
                     int force_variant, bool paged, gqa_prefill_plan* plan) {
  if (!plan) return GQA_ERR_NULL;
  std::memset(plan, 0, sizeof(*plan));
  std::vector<gqa::SeqIn> seqs;
  int total_q = 0;
  int64_t total_kv = 0;
  if (batch > 0 && !cu_seqlens_k && !kv_lens) return GQA_ERR_NULL;
  gqa_status st = gqa::batch_from_host(cu_seqlens_q, cu_seqlens_k, kv_lens, batch, &seqs,
                                       &total_q, &total_kv);
  if (st != GQA_OK) return st;
  if ((st = gqa::validate_heads(n_q_heads, n_kv_heads, head_dim, 1.0f / 16.0f)) != GQA_OK)
    return st;
  if (num_sms <= 0) return GQA_ERR_SHAPE;
  if (total_q == 0) return GQA_OK;
  // The attention calls plan with min(occupancy pairs, num_sms / 2) (device_info).
  const int pairs = max_pairs < 0 ? num_sms / 2 : std::min(max_pairs, num_sms / 2);
  gqa::cached_plan(seqs, num_sms, pairs, force_splits, force_grid, force_variant, paged, plan);
  return GQA_OK;
}
}  // namespace

gqa_status gqa_prefill_make_plan_varlen(const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                        int batch, int n_q_heads, int n_kv_heads, int head_dim,
                                        int num_sms, int max_pairs, int force_splits,
                                        int force_grid, int force_variant,
                                        gqa_prefill_plan* plan) {
  if (batch > 0 && !cu_seqlens_k) {
    if (plan) std::memset(plan, 0, sizeof(*plan));
    return GQA_ERR_NULL;
  }
  return host_plan(cu_seqlens_q, cu_seqlens_k, nullptr, batch, n_q_heads, n_kv_heads, head_dim,
                   num_sms, max_pairs, force_splits, force_grid, force_variant, false, plan);
}

gqa_status gqa_prefill_make_plan_paged_varlen(const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                                              int batch, int n_q_heads, int n_kv_heads,
                                              int head_dim, int num_sms, int max_pairs,
                                              int force_splits, int force_grid, int force_variant,
                                              gqa_prefill_plan* plan) {
  if (batch > 0 && !kv_lens) {
    if (plan) std::memset(plan, 0, sizeof(*plan));
    return GQA_ERR_NULL;
  }
  return host_plan(cu_seqlens_q, nullptr, kv_lens, batch, n_q_heads, n_kv_heads, head_dim,
                   num_sms, max_pairs, force_splits, force_grid, force_variant, true, plan);
}

gqa_status gqa_prefill_poll(void* stream, int* device_status) {
  if (!device_status) return GQA_ERR_NULL;
  gqa::DeviceInfo* dev = nullptr;
  const gqa_status st = gqa::device_info(&dev);
  if (st != GQA_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return GQA_ERR_CUDA;
  int value = 0;
  if (cudaMemcpy(&value, dev->status_word, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return GQA_ERR_CUDA;
  if (value != 0) {
    const int zero = 0;
    if (cudaMemcpy(dev->status_word, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return GQA_ERR_CUDA;
  }
  *device_status = value;
  return GQA_OK;
}

const char* gqa_status_string(gqa_status status) {
  switch (status) {
    case GQA_OK: return "ok";
    case GQA_ERR_NULL: return "a required pointer is NULL";
    case GQA_ERR_SHAPE:
      return "invalid sizes (need 0 <= q_len <= kv_len; paged: num_pages >= 1, "
             "num_pages * page_size < 2^30; FP8: k_scale_stride >= kv_len, a multiple of 4) "
             "or scale (finite, > 0)";
    case GQA_ERR_UNSUPPORTED:
      return "unsupported: needs 24 query heads, 4 KV heads, head_dim 256 on an sm_103 GPU "
             "(paged: page_size a positive multiple of 16)";
    case GQA_ERR_ALIGN: return "a tensor pointer is not 16-byte aligned";
    case GQA_ERR_CUDA: return "a CUDA call failed";
    case GQA_ERR_DEVICE_TIMEOUT: return "a device-side wait timed out; the kernel gave up";
    case GQA_ERR_SCRATCH:
      return "gqa_prefill_attn_noalloc: split partials exceed the 64 MiB static scratch "
             "(use a shorter chunk or gqa_prefill_attn)";
    case GQA_ERR_PAGE_TABLE:
      return "a block-table entry was outside [0, num_pages); that page was read as zeros";
    case GQA_ERR_BOUNDS:
      return "bounds-checked build: an output, LSE or partial-row index fell outside its buffer "
             "(the access was skipped)";
  }
  return "unknown status";
}

int gqa_prefill_abi_version(void) { return GQA_PREFILL_ABI_VERSION; }

}  // extern "C"
