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
constexpr double kMergeBytesPerUs = 3.0e6;   // effective bandwidth of the merge pass
constexpr double kMergeLaunchUs = 6.0;
constexpr int64_t kPartialRowBytes = (kHeadDim + 1) * 4;  // FP32 O row + base-2 LSE
constexpr int kSplitCandidates[] = {1, 2, 3, 4, 5, 6, 8, 10, 12, 16, 24, 32};

Geometry geometry(int q_len, int kv_len, int variant) {
  const int tpi = variant == 2 ? 2 * kTokPerTile : kTokPerTile;
  return Geometry{q_len, kv_len - q_len, (q_len + tpi - 1) / tpi, tpi};
}

// Fills *plan for `variant` (1: one CTA per item, 2: a CTA pair per item) with
// head_rounds whole rounds and S-way tail splits over `workers` CTAs (or
// pairs); S must not exceed the shortest item's tiles. Returns the estimated
// time in us.
double plan_schedule(const Geometry& geo, int num_sms, int variant, int workers, int head_rounds,
                     int S, gqa_prefill_plan* plan) {
  const int n_items = geo.n_qtiles * kKvHeads;
  const int cpi = variant == 2 ? 2 : 1;
  const int head = std::min(head_rounds * workers, n_items);
  const Schedule sc{head, S, head + (n_items - head) * S};
  workers = std::max(1, std::min(workers, sc.n_units));
  std::vector<int64_t> load(static_cast<size_t>(workers), 0);
  int64_t total = 0;
  for (int u = 0; u < sc.n_units; ++u) {
    const int r = u / workers, x = u % workers;
    const int b = (r & 1) ? workers - 1 - x : x;
    const Piece w = unit_piece(geo, sc, u);
    load[static_cast<size_t>(b)] += (w.n1 - w.n0) + kPieceOverheadTiles;
    total += w.n1 - w.n0;
  }
  const int tail = n_items - head;
  const bool split = S > 1 && tail > 0;
  std::memset(plan, 0, sizeof(*plan));
  plan->num_sms = num_sms;
  plan->q_tiles = geo.n_qtiles;
  plan->n_items = n_items;
  plan->head_rounds = head / workers;
  plan->tail_items = tail;
  plan->tail_splits = S;
  plan->n_units = sc.n_units;
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

// Best plan of one variant: searches the number of whole rounds and the tail
// split; a split must win by 2 % over the simpler plan to be taken.
double best_plan_of(int q_len, int kv_len, int num_sms, int variant, int workers, int force_splits,
                    gqa_prefill_plan* plan) {
  const Geometry geo = geometry(q_len, kv_len, variant);
  const int n_items = geo.n_qtiles * kKvHeads;
  const int max_splits = std::max(1, item_tiles(geo, 0));  // the shortest item's tiles
  const int full_rounds = n_items / workers;
  if (force_splits > 0)
    return plan_schedule(geo, num_sms, variant, workers, full_rounds,
                         std::min(force_splits, max_splits), plan);
  double best = plan_schedule(geo, num_sms, variant, workers, 0, 1, plan);  // whole items only
  gqa_prefill_plan cand{};
  for (int hr = full_rounds; hr >= 0; --hr) {
    for (int S : kSplitCandidates) {
      if (S == 1 || S > max_splits) continue;
      const double us = plan_schedule(geo, num_sms, variant, workers, hr, S, &cand);
      if (us < 0.98 * best) {
        best = us;
        *plan = cand;
      }
    }
  }
  return best;
}

// Pure function of its arguments. max_pairs: CTA pairs that can be resident at
// once. force_grid caps the CTAs launched (a pair counts as two).
void compute_plan(int q_len, int kv_len, int num_sms, int max_pairs, int force_splits,
                  int force_grid, int force_variant, gqa_prefill_plan* plan) {
  const int cap = force_grid > 0 ? std::min(force_grid, num_sms) : num_sms;
  const int workers1 = std::max(1, cap);
  const int workers2 = std::max(1, std::min(max_pairs, cap / 2));
  if (force_variant == 1 || (force_variant == 0 && max_pairs < 1)) {
    best_plan_of(q_len, kv_len, num_sms, 1, workers1, force_splits, plan);
    return;
  }
  if (force_variant == 2) {
    best_plan_of(q_len, kv_len, num_sms, 2, workers2, force_splits, plan);
    return;
  }
  gqa_prefill_plan one{}, pair{};
  const double t1 = best_plan_of(q_len, kv_len, num_sms, 1, workers1, force_splits, &one);
  const double t2 = best_plan_of(q_len, kv_len, num_sms, 2, workers2, force_splits, &pair);
  *plan = t2 < 0.98 * t1 ? pair : one;
}

struct PlanKey {
  int q_len, kv_len, num_sms, max_pairs, force_splits, force_grid, force_variant;
  bool operator<(const PlanKey& o) const {
    return std::tie(q_len, kv_len, num_sms, max_pairs, force_splits, force_grid, force_variant) <
           std::tie(o.q_len, o.kv_len, o.num_sms, o.max_pairs, o.force_splits, o.force_grid,
                    o.force_variant);
  }
};

void cached_plan(int q_len, int kv_len, int num_sms, int max_pairs, int force_splits,
                 int force_grid, int force_variant, gqa_prefill_plan* plan) {
  static std::mutex mu;
  static std::map<PlanKey, gqa_prefill_plan> cache;
  const PlanKey key{q_len, kv_len, num_sms, max_pairs, force_splits, force_grid, force_variant};
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      *plan = it->second;
      return;
    }
  }
  compute_plan(q_len, kv_len, num_sms, max_pairs, force_splits, force_grid, force_variant, plan);
  std::lock_guard<std::mutex> lock(mu);
  if (cache.size() > 4096) cache.clear();
  cache.emplace(key, *plan);
}

// --------------------------------------------------------------- validation --
gqa_status validate_shape(int q_len, int kv_len, int n_q_heads, int n_kv_heads, int head_dim,
                          float scale) {
  if (q_len < 0 || kv_len < q_len) return GQA_ERR_SHAPE;
  if (!(std::isfinite(scale) && scale > 0.0f)) return GQA_ERR_SHAPE;
  if (n_q_heads != kQHeads || n_kv_heads != kKvHeads || head_dim != kHeadDim)
    return GQA_ERR_UNSUPPORTED;
  return GQA_OK;
}

bool misaligned(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0; }

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

// A paged K or V cache [rows][4 heads][256] BF16 (rows a multiple of 16) as a
// 5-D tensor (64 d, key % 8, 64-column chunk, key / 8, head): one box of (64, 8,
// box_chunks, box_rows / 8, 1) lands in shared memory as 8-key groups, each
// holding its box_chunks chunks of 8 rows x 128 bytes — the paged stage layout
// of the attention kernel, in which a piece of whole 8-key groups is contiguous.
bool encode_kv_paged(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows,
                     uint32_t box_chunks) {
  const cuuint64_t row_bytes = static_cast<cuuint64_t>(kKvHeads) * kHeadDim * 2;
  const cuuint64_t dims[5] = {64, 8, kHeadDim / 64, rows / 8, static_cast<cuuint64_t>(kKvHeads)};
  const cuuint64_t strides[4] = {row_bytes,       // next key in the group
                                 64 * 2,          // next chunk
                                 8 * row_bytes,   // next group of 8 keys
                                 kHeadDim * 2};   // next head
  const cuuint32_t box[5] = {64, 8, box_chunks, box_rows / 8, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, base, dims, strides, box,
                CU_TENSOR_MAP_SWIZZLE_128B);
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

// Checks every argument; on success fills *plan (q_len == 0 gives an empty plan).
gqa_status check_call(const void* q, const void* k, const void* v, const void* out,
                      const float* lse, int q_len, int kv_len, int n_q_heads, int n_kv_heads,
                      int head_dim, float scale) {
  gqa_status st = validate_shape(q_len, kv_len, n_q_heads, n_kv_heads, head_dim, scale);
  if (st != GQA_OK || q_len == 0) return st;  // empty chunk: pointers may be NULL
  if (!q || !k || !v || !out) return GQA_ERR_NULL;
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(out) || misaligned(lse))
    return GQA_ERR_ALIGN;
  return GQA_OK;
}

// K/V of a paged call: the caches span num_pages * page_size rows.
struct PagedKV {
  const int32_t* block_table;
  int num_pages;
  int page_size;
};
constexpr int64_t kMaxCacheRows = int64_t{1} << 30;  // TMA row coordinates stay far from 2^31

gqa_status check_paged(const PagedKV& pkv, int q_len) {
  if (pkv.page_size <= 0 || pkv.page_size % 16 != 0) return GQA_ERR_UNSUPPORTED;
  if (pkv.num_pages < 1 || static_cast<int64_t>(pkv.num_pages) * pkv.page_size >= kMaxCacheRows)
    return GQA_ERR_SHAPE;
  if (q_len == 0) return GQA_OK;
  if (!pkv.block_table) return GQA_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(pkv.block_table) & 3u) != 0) return GQA_ERR_ALIGN;
  return GQA_OK;
}

// Quantised-QK^T inputs of a call: q and k are E4M3 codes with these scales.
struct Fp8Qk {
  const float* q_scale;  // [q_len][24]
  const float* k_scale;  // [4][k_scale_stride]
  int k_scale_stride;
};

gqa_status check_fp8(const Fp8Qk& f8, int q_len, int kv_len) {
  if (f8.k_scale_stride < kv_len || f8.k_scale_stride % 4 != 0 ||
      static_cast<int64_t>(f8.k_scale_stride) * kKvHeads >= (int64_t{1} << 31))
    return GQA_ERR_SHAPE;
  if (q_len == 0) return GQA_OK;
  if (!f8.q_scale || !f8.k_scale) return GQA_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(f8.q_scale) & 3u) != 0 || misaligned(f8.k_scale))
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

// Launches `plan` on `stream`; `ws` holds plan.workspace_bytes (or nothing).
// `pkv` is null for dense K/V, otherwise k and v are the paged caches; `f8` is
// null for BF16 Q/K, otherwise q and k are E4M3 codes with its scales.
gqa_status launch_plan(const gqa_prefill_plan& plan, const void* q, const void* k, const void* v,
                       const PagedKV* pkv, const Fp8Qk* f8, void* out, float* lse, int q_len,
                       int kv_len, float scale, int* status_word, void* ws,
                       const gqa_prefill_opts* opts, cudaStream_t stream) {
  const bool pair = plan.variant == 2;
  if (pkv && f8) return GQA_ERR_UNSUPPORTED;
  FwdParams p;
  std::memset(&p, 0, sizeof(p));
  const uint64_t kv_rows = pkv ? static_cast<uint64_t>(pkv->num_pages) * pkv->page_size
                               : static_cast<uint64_t>(kv_len);
  const Elem qk = f8 ? kE4m3 : kBf16;
  // K/V stages per CTA: one-CTA K 128 keys (BF16: 2 chunks per stage, 2 stages;
  // FP8: all 2 chunks), V 64 keys x 4 chunks; pairs K 64 keys x all chunks,
  // V 128 keys x 2 chunks.
  const uint32_t k_rows = pair ? 64 : kBlockN;
  const uint32_t k_chunks = f8 ? 2 : (pair ? 4 : 2);
  const uint32_t v_rows = pair ? kBlockN : 64, v_chunks = pair ? 2 : 4;
  if (!encode_q(&p.tmap_q, q, static_cast<uint64_t>(q_len), qk)) return GQA_ERR_CUDA;
  p.v_fix_tile = -1;
  if (!pkv) {
    if (!encode_kv(&p.tmap_k, k, kv_rows, k_rows, k_chunks, qk) ||
        !encode_kv(&p.tmap_v, v, kv_rows, v_rows, v_chunks, kBf16))
      return GQA_ERR_CUDA;
  } else {
    const uint32_t sub = static_cast<uint32_t>(gcd_int(pkv->page_size, 64));  // 16, 32 or 64
    if (!encode_kv_paged(&p.tmap_k, k, kv_rows, k_rows, k_chunks) ||
        !encode_kv_paged(&p.tmap_v, v, kv_rows, v_rows, v_chunks) ||
        !encode_kv_paged(&p.tmap_k_sub, k, kv_rows, sub, k_chunks) ||
        !encode_kv_paged(&p.tmap_v_sub, v, kv_rows, sub, v_chunks) ||
        !encode_kv_paged(&p.tmap_v16, v, kv_rows, 16, v_chunks))
      return GQA_ERR_CUDA;
    p.block_table = pkv->block_table;
    p.page_size = pkv->page_size;
    p.num_pages = pkv->num_pages;
    p.sub_rows = static_cast<int>(sub);
    p.oob_row = static_cast<int>(kv_rows);
    if (kv_len % kBlockN != 0) p.v_fix_tile = (kv_len - 1) / kBlockN;
  }
  if (f8) {
    if (!encode_key_scales(&p.tmap_ks, f8->k_scale, static_cast<uint64_t>(kv_len),
                           static_cast<uint64_t>(f8->k_scale_stride)))
      return GQA_ERR_CUDA;
    p.q_scale = f8->q_scale;
  }
  const int workers = pair ? plan.grid / 2 : plan.grid;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.status = status_word;
  p.q_len = q_len;
  p.kv_len = kv_len;
  p.p0 = kv_len - q_len;
  p.n_qtiles = plan.q_tiles;
  p.head_items = std::min(plan.head_rounds * workers, plan.n_items);
  p.tail_splits = plan.tail_splits;
  p.n_units = plan.n_units;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.timeout_ns = (opts && opts->wait_timeout_us) ? 1000ull * opts->wait_timeout_us
                                                 : kDefaultTimeoutNs;
  p.withhold_q = (opts && opts->test_withhold_q) ? 1 : 0;
  if (plan.kernels_per_call == 2) {
    p.part_o = static_cast<float*>(ws);
    p.part_lse = p.part_o + static_cast<size_t>(plan.tail_items) * plan.tail_splits *
                                (pair ? 2 : 1) * kRowsPerTile * kHeadDim;
  }
  auto ev_begin = static_cast<cudaEvent_t>(opts ? opts->fwd_event_begin : nullptr);
  auto ev_end = static_cast<cudaEvent_t>(opts ? opts->fwd_event_end : nullptr);
  if (ev_begin && cudaEventRecord(ev_begin, stream) != cudaSuccess) return GQA_ERR_CUDA;
  if (launch_fwd(p, plan.grid, pair, pkv != nullptr, f8 != nullptr, stream) != cudaSuccess)
    return GQA_ERR_CUDA;
  if (ev_end && cudaEventRecord(ev_end, stream) != cudaSuccess) return GQA_ERR_CUDA;
  if (plan.kernels_per_call == 2) {
    MergeParams m{p.part_o, p.part_lse, p.out, lse, q_len, p.n_qtiles, p.head_items,
                  plan.tail_items, plan.tail_splits, pair ? 2 : 1};
    if (launch_merge(m, stream) != cudaSuccess) return GQA_ERR_CUDA;
  }
  return GQA_OK;
}

gqa_status run(const void* q, const void* k, const void* v, const PagedKV* pkv, const Fp8Qk* f8,
               void* out, float* lse, int q_len, int kv_len, int n_q_heads, int n_kv_heads,
               int head_dim, float scale, void* stream_ptr, const gqa_prefill_opts* opts,
               gqa_prefill_plan* plan_out) {
  if (plan_out) std::memset(plan_out, 0, sizeof(*plan_out));
  gqa_status st = check_call(q, k, v, out, lse, q_len, kv_len, n_q_heads, n_kv_heads, head_dim, scale);
  if (st == GQA_OK && pkv) st = check_paged(*pkv, q_len);
  if (st == GQA_OK && f8) st = check_fp8(*f8, q_len, kv_len);
  if (st != GQA_OK || q_len == 0) return st;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != GQA_OK) return st;
  gqa_prefill_plan plan{};
  cached_plan(q_len, kv_len, dev->num_sms, dev->max_pairs, opts ? opts->force_splits : 0,
              opts ? opts->force_grid : 0, opts ? opts->force_variant : 0, &plan);
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
  st = launch_plan(plan, q, k, v, pkv, f8, out, lse, q_len, kv_len, scale, dev->status_word, ws,
                   opts, stream);
  if (ws && cudaFreeAsync(ws, stream) != cudaSuccess) st = GQA_ERR_CUDA;
  return st;
}

// ---------------------------------------------------- allocation-free variant --
// Split-KV partials of gqa_prefill_attn_noalloc live in this file-scope array
// instead of the stream-ordered pool. In host code `g_noalloc_scratch` is only a
// host-side stand-in for the symbol: its device address comes from
// cudaGetSymbolAddress, once per device, with that device current.
constexpr size_t kNoAllocScratchBytes = GQA_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocDeviceState {
  std::once_flag once;
  gqa_status status = GQA_OK;
  void* scratch = nullptr;  // device address of g_noalloc_scratch on this device
};
NoAllocDeviceState g_noalloc_dev[kMaxDevices];

gqa_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GQA_ERR_CUDA;
  NoAllocDeviceState& s = g_noalloc_dev[dev];
  std::call_once(s.once, [&s] {
    if (cudaGetSymbolAddress(&s.scratch, g_noalloc_scratch) != cudaSuccess || s.scratch == nullptr)
      s.status = GQA_ERR_CUDA;
  });
  if (s.status != GQA_OK) return s.status;
  *out = s.scratch;
  return GQA_OK;
}

gqa_status run_noalloc(const void* q, const void* k, const void* v, void* out, float* lse,
                       int q_len, int kv_len, int n_q_heads, int n_kv_heads, int head_dim,
                       float scale, void* stream_ptr) {
  gqa_status st = check_call(q, k, v, out, lse, q_len, kv_len, n_q_heads, n_kv_heads, head_dim, scale);
  if (st != GQA_OK || q_len == 0) return st;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != GQA_OK) return st;
  void* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != GQA_OK) return st;
  gqa_prefill_plan plan{};
  cached_plan(q_len, kv_len, dev->num_sms, dev->max_pairs, 0, 0, 0, &plan);
  if (static_cast<uint64_t>(plan.workspace_bytes) > kNoAllocScratchBytes) return GQA_ERR_SCRATCH;
  // Every partial row the merge reads is written by the attention kernel first,
  // so the scratch needs no clearing between calls.
  return launch_plan(plan, q, k, v, nullptr, nullptr, out, lse, q_len, kv_len, scale,
                     dev->status_word, scratch, nullptr, static_cast<cudaStream_t>(stream_ptr));
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
  return gqa::run(q, k, v, nullptr, nullptr, out, lse, q_len, kv_len, n_q_heads, n_kv_heads,
                  head_dim, scale, stream, nullptr, nullptr);
}

gqa_status gqa_prefill_attn_ex(const void* q, const void* k, const void* v, void* out, float* lse,
                               int q_len, int kv_len, int n_q_heads, int n_kv_heads, int head_dim,
                               float scale, void* stream, const gqa_prefill_opts* opts,
                               gqa_prefill_plan* plan_out) {
  return gqa::run(q, k, v, nullptr, nullptr, out, lse, q_len, kv_len, n_q_heads, n_kv_heads,
                  head_dim, scale, stream, opts, plan_out);
}

gqa_status gqa_prefill_attn_paged(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_table, int num_pages, int page_size,
                                  void* out, float* lse, int q_len, int kv_len, int n_q_heads,
                                  int n_kv_heads, int head_dim, float scale, void* stream) {
  const gqa::PagedKV pkv{block_table, num_pages, page_size};
  return gqa::run(q, k_cache, v_cache, &pkv, nullptr, out, lse, q_len, kv_len, n_q_heads,
                  n_kv_heads, head_dim, scale, stream, nullptr, nullptr);
}

gqa_status gqa_prefill_attn_paged_ex(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_table, int num_pages, int page_size,
                                     void* out, float* lse, int q_len, int kv_len,
                                     int n_q_heads, int n_kv_heads, int head_dim, float scale,
                                     void* stream, const gqa_prefill_opts* opts,
                                     gqa_prefill_plan* plan_out) {
  const gqa::PagedKV pkv{block_table, num_pages, page_size};
  return gqa::run(q, k_cache, v_cache, &pkv, nullptr, out, lse, q_len, kv_len, n_q_heads,
                  n_kv_heads, head_dim, scale, stream, opts, plan_out);
}

gqa_status gqa_quantize_q_fp8(const void* q, void* q_fp8, float* q_scale, int q_len,
                              int n_q_heads, int head_dim, void* stream) {
  if (q_len < 0) return GQA_ERR_SHAPE;
  if (n_q_heads != gqa::kQHeads || head_dim != gqa::kHeadDim) return GQA_ERR_UNSUPPORTED;
  if (q_len == 0) return GQA_OK;
  if (!q || !q_fp8 || !q_scale) return GQA_ERR_NULL;
  if (gqa::misaligned(q) || gqa::misaligned(q_fp8) || (reinterpret_cast<uintptr_t>(q_scale) & 3u))
    return GQA_ERR_ALIGN;
  return gqa::launch_quantize_fp8(q, q_fp8, q_scale, q_len, gqa::kQHeads, 0, false,
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
  return gqa::launch_quantize_fp8(k, k_fp8, k_scale, kv_len, gqa::kKvHeads, k_scale_stride, true,
                                  static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? GQA_OK
             : GQA_ERR_CUDA;
}

gqa_status gqa_prefill_attn_fp8qk(const void* q_fp8, const float* q_scale, const void* k_fp8,
                                  const float* k_scale, int k_scale_stride, const void* v,
                                  void* out, float* lse, int q_len, int kv_len, int n_q_heads,
                                  int n_kv_heads, int head_dim, float scale, void* stream) {
  const gqa::Fp8Qk f8{q_scale, k_scale, k_scale_stride};
  return gqa::run(q_fp8, k_fp8, v, nullptr, &f8, out, lse, q_len, kv_len, n_q_heads, n_kv_heads,
                  head_dim, scale, stream, nullptr, nullptr);
}

gqa_status gqa_prefill_attn_fp8qk_ex(const void* q_fp8, const float* q_scale, const void* k_fp8,
                                     const float* k_scale, int k_scale_stride, const void* v,
                                     void* out, float* lse, int q_len, int kv_len, int n_q_heads,
                                     int n_kv_heads, int head_dim, float scale, void* stream,
                                     const gqa_prefill_opts* opts, gqa_prefill_plan* plan_out) {
  const gqa::Fp8Qk f8{q_scale, k_scale, k_scale_stride};
  return gqa::run(q_fp8, k_fp8, v, nullptr, &f8, out, lse, q_len, kv_len, n_q_heads, n_kv_heads,
                  head_dim, scale, stream, opts, plan_out);
}

gqa_status gqa_prefill_make_plan(int q_len, int kv_len, int n_q_heads, int n_kv_heads, int head_dim,
                                 int num_sms, int force_splits, int force_grid, int force_variant,
                                 gqa_prefill_plan* plan) {
  if (!plan) return GQA_ERR_NULL;
  const gqa_status st =
      gqa::validate_shape(q_len, kv_len, n_q_heads, n_kv_heads, head_dim, 1.0f / 16.0f);
  if (st != GQA_OK) return st;
  if (num_sms <= 0) return GQA_ERR_SHAPE;
  std::memset(plan, 0, sizeof(*plan));
  if (q_len == 0) return GQA_OK;
  gqa::cached_plan(q_len, kv_len, num_sms, num_sms / 2, force_splits, force_grid, force_variant,
                   plan);
  return GQA_OK;
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
  }
  return "unknown status";
}

int gqa_prefill_abi_version(void) { return GQA_PREFILL_ABI_VERSION; }

}  // extern "C"
