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
// 128 x 128 x 256 block: ~1.3 us of tensor-core time on one SM at peak).
constexpr int64_t kPieceOverheadTiles = 2;   // Q load, pipeline fill, epilogue
constexpr double kTileUs = 1.5;              // planning estimate per tile
constexpr double kMergeBytesPerUs = 6.0e6;   // HBM bandwidth for the merge pass
constexpr double kMergeLaunchUs = 4.0;
constexpr int64_t kPartialRowBytes = (kHeadDim + 1) * 4;  // FP32 O row + base-2 LSE
constexpr int kSplitCandidates[] = {1, 2, 3, 4, 5, 6, 8, 10, 12, 16};

Geometry geometry(int q_len, int kv_len) {
  return Geometry{q_len, kv_len - q_len, (q_len + kTokPerTile - 1) / kTokPerTile};
}

// Fills *plan for head_rounds whole rounds and S-way tail splits on `grid` CTAs
// (S must not exceed the shortest item's tiles); returns the estimated time in us.
double plan_schedule(const Geometry& geo, int num_sms, int grid, int head_rounds, int S,
                     gqa_prefill_plan* plan) {
  const int n_items = geo.n_qtiles * kKvHeads;
  const int head = std::min(head_rounds * grid, n_items);
  const Schedule sc{head, S, head + (n_items - head) * S};
  grid = std::max(1, std::min(grid, sc.n_units));
  std::vector<int64_t> load(static_cast<size_t>(grid), 0);
  int64_t total = 0;
  for (int u = 0; u < sc.n_units; ++u) {
    const int r = u / grid, x = u % grid;
    const int b = (r & 1) ? grid - 1 - x : x;
    const Piece w = unit_piece(geo, sc, u);
    load[static_cast<size_t>(b)] += (w.n1 - w.n0) + kPieceOverheadTiles;
    total += w.n1 - w.n0;
  }
  const int tail = n_items - head;
  std::memset(plan, 0, sizeof(*plan));
  plan->num_sms = num_sms;
  plan->q_tiles = geo.n_qtiles;
  plan->n_items = n_items;
  plan->head_rounds = head / grid;
  plan->tail_items = tail;
  plan->tail_splits = S;
  plan->n_units = sc.n_units;
  plan->grid = grid;
  plan->kernels_per_call = (S > 1 && tail > 0) ? 2 : 1;
  plan->variant = 1;
  plan->total_tiles = total;
  plan->workspace_bytes =
      (S > 1 && tail > 0) ? static_cast<int64_t>(tail) * S * kRowsPerTile * kPartialRowBytes : 0;
  plan->est_makespan_tiles = *std::max_element(load.begin(), load.end());
  double us = static_cast<double>(plan->est_makespan_tiles) * kTileUs;
  if (plan->kernels_per_call == 2) {
    const double bytes = tail * static_cast<double>(kRowsPerTile) * (S * kPartialRowBytes + 520.0);
    us += bytes / kMergeBytesPerUs + kMergeLaunchUs;
  }
  return us;
}

// Pure function of its arguments. Searches the number of whole rounds and the
// tail split; a split must win by 2 % over the simpler plan to be taken.
void compute_plan(int q_len, int kv_len, int num_sms, int force_splits, int force_grid,
                  gqa_prefill_plan* plan) {
  const Geometry geo = geometry(q_len, kv_len);
  const int n_items = geo.n_qtiles * kKvHeads;
  const int grid = std::max(1, force_grid > 0 ? std::min(force_grid, num_sms) : num_sms);
  const int max_splits = std::max(1, item_tiles(geo, 0));  // the shortest item's tiles
  const int full_rounds = n_items / grid;
  if (force_splits > 0) {
    plan_schedule(geo, num_sms, grid, full_rounds, std::min(force_splits, max_splits), plan);
    return;
  }
  double best = plan_schedule(geo, num_sms, grid, 0, 1, plan);  // whole items only
  gqa_prefill_plan cand{};
  for (int hr = full_rounds; hr >= 0; --hr) {
    for (int S : kSplitCandidates) {
      if (S == 1 || S > max_splits) continue;
      const double us = plan_schedule(geo, num_sms, grid, hr, S, &cand);
      if (us < 0.98 * best) {
        best = us;
        *plan = cand;
      }
    }
  }
}

struct PlanKey {
  int q_len, kv_len, num_sms, force_splits, force_grid;
  bool operator<(const PlanKey& o) const {
    return std::tie(q_len, kv_len, num_sms, force_splits, force_grid) <
           std::tie(o.q_len, o.kv_len, o.num_sms, o.force_splits, o.force_grid);
  }
};

void cached_plan(int q_len, int kv_len, int num_sms, int force_splits, int force_grid,
                 gqa_prefill_plan* plan) {
  static std::mutex mu;
  static std::map<PlanKey, gqa_prefill_plan> cache;
  const PlanKey key{q_len, kv_len, num_sms, force_splits, force_grid};
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      *plan = it->second;
      return;
    }
  }
  compute_plan(q_len, kv_len, num_sms, force_splits, force_grid, plan);
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
struct DeviceState {
  std::once_flag once;
  cudaError_t init_err = cudaSuccess;
  bool supported = false;
  int num_sms = 0;
  int* status = nullptr;
  cudaMemPool_t pool = nullptr;
};
DeviceState g_dev[kMaxDevices];

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

gqa_status device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GQA_ERR_CUDA;
  DeviceState& s = g_dev[dev];
  std::call_once(s.once, [&s, dev] {
    cudaDeviceProp prop{};
    if ((s.init_err = cudaGetDeviceProperties(&prop, dev)) != cudaSuccess) return;
    // The kernels are built for sm_103a only (tcgen05 / TMEM / TMA).
    s.supported = prop.major == 10 && prop.minor == 3;
    s.num_sms = prop.multiProcessorCount;
    if (!s.supported) return;
    if ((s.init_err = prepare_fwd_kernel()) != cudaSuccess) return;
    if ((s.init_err = status_word_address(&s.status)) != cudaSuccess) return;
    cudaMemPoolProps props{};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    if ((s.init_err = cudaMemPoolCreate(&s.pool, &props)) != cudaSuccess) return;
    uint64_t keep = UINT64_MAX;  // keep freed partial buffers cached in the pool
    s.init_err = cudaMemPoolSetAttribute(s.pool, cudaMemPoolAttrReleaseThreshold, &keep);
  });
  if (s.init_err != cudaSuccess) return GQA_ERR_CUDA;
  if (!s.supported) return GQA_ERR_UNSUPPORTED;
  *out = &s;
  return GQA_OK;
}

bool encode_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
               uint32_t b0, uint32_t b1, uint32_t b2) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};  // bytes, dims 1 and 2
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

gqa_status run(const void* q, const void* k, const void* v, void* out, float* lse, int q_len,
               int kv_len, int n_q_heads, int n_kv_heads, int head_dim, float scale, void* stream_ptr,
               const gqa_prefill_opts* opts, gqa_prefill_plan* plan_out) {
  gqa_status st = validate_shape(q_len, kv_len, n_q_heads, n_kv_heads, head_dim, scale);
  if (st != GQA_OK) return st;
  if (q_len == 0) {
    if (plan_out) std::memset(plan_out, 0, sizeof(*plan_out));
    return GQA_OK;  // empty chunk: nothing to compute, pointers may be NULL
  }
  if (!q || !k || !v || !out) return GQA_ERR_NULL;
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(out) || misaligned(lse))
    return GQA_ERR_ALIGN;
  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != GQA_OK) return st;

  gqa_prefill_plan plan{};
  cached_plan(q_len, kv_len, dev->num_sms, opts ? opts->force_splits : 0,
              opts ? opts->force_grid : 0, &plan);
  if (plan_out) *plan_out = plan;

  auto stream = static_cast<cudaStream_t>(stream_ptr);
  FwdParams p;
  std::memset(&p, 0, sizeof(p));
  if (!encode_3d(&p.tmap_q, q, kHeadDim, kQHeads, static_cast<uint64_t>(q_len), 64, kGroup,
                 kTokPerTile) ||
      !encode_3d(&p.tmap_k, k, kHeadDim, kKvHeads, static_cast<uint64_t>(kv_len), 64, 1, kBlockN) ||
      !encode_3d(&p.tmap_v, v, kHeadDim, kKvHeads, static_cast<uint64_t>(kv_len), 64, 1, 64))
    return GQA_ERR_CUDA;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.status = dev->status;
  p.q_len = q_len;
  p.kv_len = kv_len;
  p.p0 = kv_len - q_len;
  p.n_qtiles = plan.q_tiles;
  p.head_items = plan.head_rounds * plan.grid < plan.n_items ? plan.head_rounds * plan.grid
                                                             : plan.n_items;
  p.tail_splits = plan.tail_splits;
  p.n_units = plan.n_units;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.timeout_ns = (opts && opts->wait_timeout_us) ? 1000ull * opts->wait_timeout_us
                                                 : kDefaultTimeoutNs;
  p.withhold_q = (opts && opts->test_withhold_q) ? 1 : 0;

  void* ws = nullptr;
  const size_t n_slots = static_cast<size_t>(plan.tail_items) * plan.tail_splits;
  if (plan.kernels_per_call == 2) {
    if (cudaMallocFromPoolAsync(&ws, static_cast<size_t>(plan.workspace_bytes), dev->pool, stream) !=
        cudaSuccess)
      return GQA_ERR_CUDA;
    p.part_o = static_cast<float*>(ws);
    p.part_lse = p.part_o + n_slots * kRowsPerTile * kHeadDim;
  }
  auto ev_begin = static_cast<cudaEvent_t>(opts ? opts->fwd_event_begin : nullptr);
  auto ev_end = static_cast<cudaEvent_t>(opts ? opts->fwd_event_end : nullptr);
  if (ev_begin && cudaEventRecord(ev_begin, stream) != cudaSuccess) st = GQA_ERR_CUDA;
  if (st == GQA_OK && launch_fwd(p, plan.grid, stream) != cudaSuccess) st = GQA_ERR_CUDA;
  if (st == GQA_OK && ev_end && cudaEventRecord(ev_end, stream) != cudaSuccess) st = GQA_ERR_CUDA;
  if (st == GQA_OK && plan.kernels_per_call == 2) {
    MergeParams m{p.part_o, p.part_lse, p.out, lse, q_len, p.n_qtiles, p.head_items,
                  plan.tail_items, plan.tail_splits};
    if (launch_merge(m, stream) != cudaSuccess) st = GQA_ERR_CUDA;
  }
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
  int num_sms = 0;
  int* status_word = nullptr;
  void* scratch = nullptr;  // device address of g_noalloc_scratch on this device
};
NoAllocDeviceState g_noalloc_dev[kMaxDevices];

gqa_status noalloc_device_state(NoAllocDeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GQA_ERR_CUDA;
  NoAllocDeviceState& s = g_noalloc_dev[dev];
  std::call_once(s.once, [&s, dev] {
    cudaDeviceProp prop{};
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) { s.status = GQA_ERR_CUDA; return; }
    if (!(prop.major == 10 && prop.minor == 3)) { s.status = GQA_ERR_UNSUPPORTED; return; }
    s.num_sms = prop.multiProcessorCount;
    if (prepare_fwd_kernel() != cudaSuccess || status_word_address(&s.status_word) != cudaSuccess ||
        cudaGetSymbolAddress(&s.scratch, g_noalloc_scratch) != cudaSuccess || s.scratch == nullptr) {
      s.status = GQA_ERR_CUDA;
      return;
    }
  });
  if (s.status != GQA_OK) return s.status;
  *out = &s;
  return GQA_OK;
}

gqa_status run_noalloc(const void* q, const void* k, const void* v, void* out, float* lse,
                       int q_len, int kv_len, int n_q_heads, int n_kv_heads, int head_dim,
                       float scale, void* stream_ptr) {
  gqa_status st = validate_shape(q_len, kv_len, n_q_heads, n_kv_heads, head_dim, scale);
  if (st != GQA_OK) return st;
  if (q_len == 0) return GQA_OK;
  if (!q || !k || !v || !out) return GQA_ERR_NULL;
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(out) || misaligned(lse))
    return GQA_ERR_ALIGN;
  NoAllocDeviceState* dev = nullptr;
  if ((st = noalloc_device_state(&dev)) != GQA_OK) return st;
  gqa_prefill_plan plan{};
  cached_plan(q_len, kv_len, dev->num_sms, 0, 0, &plan);
  if (static_cast<uint64_t>(plan.workspace_bytes) > kNoAllocScratchBytes) return GQA_ERR_SCRATCH;

  auto stream = static_cast<cudaStream_t>(stream_ptr);
  FwdParams p;
  std::memset(&p, 0, sizeof(p));
  if (!encode_3d(&p.tmap_q, q, kHeadDim, kQHeads, static_cast<uint64_t>(q_len), 64, kGroup,
                 kTokPerTile) ||
      !encode_3d(&p.tmap_k, k, kHeadDim, kKvHeads, static_cast<uint64_t>(kv_len), 64, 1, kBlockN) ||
      !encode_3d(&p.tmap_v, v, kHeadDim, kKvHeads, static_cast<uint64_t>(kv_len), 64, 1, 64))
    return GQA_ERR_CUDA;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.status = dev->status_word;
  p.q_len = q_len;
  p.kv_len = kv_len;
  p.p0 = kv_len - q_len;
  p.n_qtiles = plan.q_tiles;
  p.head_items = plan.head_rounds * plan.grid < plan.n_items ? plan.head_rounds * plan.grid
                                                             : plan.n_items;
  p.tail_splits = plan.tail_splits;
  p.n_units = plan.n_units;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.timeout_ns = kDefaultTimeoutNs;
  if (plan.kernels_per_call == 2) {
    // Every partial row the merge reads is written by the attention kernel first,
    // so the scratch needs no clearing between calls.
    p.part_o = static_cast<float*>(dev->scratch);
    p.part_lse = p.part_o + static_cast<size_t>(plan.tail_items) * plan.tail_splits *
                                kRowsPerTile * kHeadDim;
  }
  if (launch_fwd(p, plan.grid, stream) != cudaSuccess) return GQA_ERR_CUDA;
  if (plan.kernels_per_call == 2) {
    MergeParams m{p.part_o, p.part_lse, p.out, lse, q_len, p.n_qtiles, p.head_items,
                  plan.tail_items, plan.tail_splits};
    if (launch_merge(m, stream) != cudaSuccess) return GQA_ERR_CUDA;
  }
  return GQA_OK;
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
  return gqa::run(q, k, v, out, lse, q_len, kv_len, n_q_heads, n_kv_heads, head_dim, scale, stream,
                  nullptr, nullptr);
}

gqa_status gqa_prefill_attn_ex(const void* q, const void* k, const void* v, void* out, float* lse,
                               int q_len, int kv_len, int n_q_heads, int n_kv_heads, int head_dim,
                               float scale, void* stream, const gqa_prefill_opts* opts,
                               gqa_prefill_plan* plan_out) {
  return gqa::run(q, k, v, out, lse, q_len, kv_len, n_q_heads, n_kv_heads, head_dim, scale, stream,
                  opts, plan_out);
}

gqa_status gqa_prefill_make_plan(int q_len, int kv_len, int n_q_heads, int n_kv_heads, int head_dim,
                                 int num_sms, int force_splits, int force_grid,
                                 gqa_prefill_plan* plan) {
  if (!plan) return GQA_ERR_NULL;
  const gqa_status st =
      gqa::validate_shape(q_len, kv_len, n_q_heads, n_kv_heads, head_dim, 1.0f / 16.0f);
  if (st != GQA_OK) return st;
  if (num_sms <= 0) return GQA_ERR_SHAPE;
  std::memset(plan, 0, sizeof(*plan));
  if (q_len == 0) return GQA_OK;
  gqa::cached_plan(q_len, kv_len, num_sms, force_splits, force_grid, plan);
  return GQA_OK;
}

gqa_status gqa_prefill_poll(void* stream, int* device_status) {
  if (!device_status) return GQA_ERR_NULL;
  gqa::DeviceState* dev = nullptr;
  const gqa_status st = gqa::device_state(&dev);
  if (st != GQA_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return GQA_ERR_CUDA;
  int value = 0;
  if (cudaMemcpy(&value, dev->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return GQA_ERR_CUDA;
  if (value != 0) {
    const int zero = 0;
    if (cudaMemcpy(dev->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return GQA_ERR_CUDA;
  }
  *device_status = value;
  return GQA_OK;
}

const char* gqa_status_string(gqa_status status) {
  switch (status) {
    case GQA_OK: return "ok";
    case GQA_ERR_NULL: return "a required pointer is NULL";
    case GQA_ERR_SHAPE: return "invalid sizes (need 0 <= q_len <= kv_len) or scale (finite, > 0)";
    case GQA_ERR_UNSUPPORTED:
      return "unsupported: needs 24 query heads, 4 KV heads, head_dim 256 on an sm_103 GPU";
    case GQA_ERR_ALIGN: return "a tensor pointer is not 16-byte aligned";
    case GQA_ERR_CUDA: return "a CUDA call failed";
    case GQA_ERR_DEVICE_TIMEOUT: return "a device-side wait timed out; the kernel gave up";
    case GQA_ERR_SCRATCH:
      return "gqa_prefill_attn_noalloc: split partials exceed the 64 MiB static scratch "
             "(use a shorter chunk or gqa_prefill_attn)";
  }
  return "unknown status";
}

int gqa_prefill_abi_version(void) { return GQA_PREFILL_ABI_VERSION; }

}  // extern "C"
