// Chunked-prefill causal GQA attention forward for GB300 (sm_103a).
//
// Method (DCU使用技术报告（中篇）：gfx936 DCU上的Qwen3.5-27B Triton-ROCm Attention与
// GEMV深度优化实战, §2): QK^T, causal mask, online softmax, PV, FP32 accumulation,
// one sequence, 24 query heads / 4 KV heads / head_dim 256.
//
// GB300 design (what differs from the report's Triton kernels for gfx936):
//  * GQA in the MMA M dimension. The report packs 5 tokens x 6 heads = 30 of 32
//    rows (§2) and then enlarges the query block per K/V fetch (§4 "Q10", §5
//    "Q20") so one K/V tile serves more queries. Here one 128-row tcgen05 MMA
//    tile holds 21 tokens x 6 heads = 126 rows of one KV group, loaded by a
//    single 3-D TMA box per 64-wide d chunk; rows 126/127 are idle (zeroed,
//    never stored). Every K/V tile is fetched once per 126 query rows.
//  * The report's two-stage KV software pipeline with a delayed V load (§3)
//    becomes five 32 KB shared-memory stages fed by TMA and tracked by
//    mbarriers, split into a K ring and a V ring (one reader each); K of tile
//    j+2 streams while V of tile j is used.
//  * S = Q K^T and O += P V are tcgen05 MMAs (kind::f16, BF16 in, FP32 out).
//    Tensor memory (512 columns) holds O (128 x 256 FP32), one S tile
//    (128 x 128 FP32) and two BF16 P tiles (64 columns each) that feed the PV
//    MMA straight from tensor memory. No MMA ever writes columns that another
//    in-flight MMA reads: the next QK^T may overwrite S as soon as the softmax
//    has copied S into registers (s_free), and P[b] is rewritten only after
//    the PV that read it has completed (pv_done[b]). tcgen05 only orders
//    consecutive MMAs that share accumulator and shape, so these two barriers
//    are what makes the S -> QK^T and P -> PV reuse safe.
//  * Warp specialisation: one warp issues TMA (two, one per ring, on paged
//    K/V), two issue MMAs (one thread each: QK^T and PV,
//    so that one keeps the tensor pipe fed while the other waits on a
//    barrier), and the softmax warps take the MMA rows (tensor-memory lanes). BF16 and FP8 QK^T: warps 0-3, one thread per row, so row max and
//    row sum need no cross-thread reduction. Quantised PV, where the softmax
//    (not the tensor core) sets the pace: warps 0-7, two threads per row on 64
//    keys of each tile each, which trade the row's tile maximum through shared
//    memory; two warps per scheduler hide each other's latencies.
//  * Online softmax in base 2 with the scale folded into one FMA. O is only
//    rescaled when a row's running max grows by more than 2^8; otherwise the
//    stale max is kept, which is exact after the final division by the row sum.
//  * Causal tiles entirely above the diagonal are never visited; only the (at
//    most two) tiles that straddle it are masked element-wise.
//  * Persistent grid (one CTA per SM). Work items (query tile, KV group) are
//    ordered longest first and dealt out in a snake, whole items in full
//    rounds; the items of the last, partial round are split along KV into
//    equal pieces so that they spread over all CTAs (gqa_schedule.h). Each
//    piece writes a normalised FP32 partial plus its base-2 LSE, and
//    merge_tail_kernel (a warp per row) or, for items of 16 pieces or more,
//    merge_wide_kernel (a block per row) combines them.
//  * Every mbarrier wait is bounded: on time-out the kernel records
//    GQA_ERR_DEVICE_TIMEOUT, waits for its own TMA copies in flight, frees its
//    tensor memory and returns.

#include <algorithm>

#include "gqa_internal.h"
#include "gqa_paged.h"
#include "gqa_prefill.h"
#include "gqa_schedule.h"
#include "sm100_ptx.cuh"

namespace gqa {

namespace {

constexpr int kStages = 5;
// A compile-time flag as a value (selects a generic lambda's instantiation).
template <bool B>
struct BoolC {
  static constexpr bool value = B;
};
constexpr uint32_t kQChunkBytes = 128 * 128;   // 128 rows x 64 bf16 (one 128B-swizzle column)
constexpr uint32_t kQBoxBytes = 126 * 128;     // the 21x6 rows one TMA box writes
constexpr uint32_t kQBytes = 4 * kQChunkBytes;  // d = 256 -> 4 chunks
constexpr uint32_t kStageBytes = 32768;

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;    // O: 256 FP32 columns
constexpr uint32_t kTmemS = 256;  // S: 128 FP32 columns
constexpr uint32_t kTmemP = 384;  // P buffer b: 64 columns of packed BF16 pairs at kTmemP + 64*b

// Shared-memory map (offsets from a 1024-byte aligned base).
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffStages = kOffQ + kQBytes;
constexpr uint32_t kOffBars = kOffStages + kStages * kStageBytes;
enum BarId : uint32_t {
  kBarFull = 0,                 // [kStages] stage loaded (TMA tx)
  kBarEmpty = kStages,          // [kStages] stage consumed (MMA commit)
  kBarQFull = 2 * kStages,      // Q tile loaded
  kBarQEmpty,                   // last QK^T of the unit done with Q
  kBarSFull,                    // S holds a finished QK^T (MMA commit)
  kBarSFree,                    // softmax copied S to registers (128 arrivals)
  kBarPFull0,                   // [2] P[b] written, O corrected (128 arrivals)
  kBarPFull1,
  kBarPvDone0,                  // [2] the PV that read P[b] completed (MMA commit)
  kBarPvDone1,
  kBarOFree,                    // epilogue finished reading O (128 arrivals)
  kBarDrain,                    // the MMA threads' final drain (2 commits)
  kBarScFull,                   // [kScSlots] FP8 QK^T: key scales of a tile loaded (TMA tx)
  kBarScEmpty = kBarScFull + 8, // [kScSlots] this CTA's softmax done with them (all its softmax threads)
  kBarXch = kBarScEmpty + 8,    // [4] FP8: the two softmax threads of each row of a 32-row
                                //   quarter traded a value (64 arrivals)
  kNumBars = kBarXch + 4
};
// FP8 QK^T: Q codes take 2 of the 4 Q chunks; the key-scale ring (one 128-key
// FP32 row per slot, consumed by the softmax warps) lives in the other half.
constexpr int kScSlots = 8;
constexpr uint32_t kScSlotBytes = 128 * 4;
constexpr uint32_t kOffScales = kOffQ + 2 * kQChunkBytes;
// FP8: the values the two softmax threads of a row trade (two slots x two
// halves x 128 rows of FP32), after the key-scale ring.
constexpr uint32_t kOffXch = kOffScales + kScSlots * kScSlotBytes;
static_assert(kOffXch + 2 * 2 * 128 * 4 <= kOffQ + kQBytes, "exchange slots fit beside the FP8 Q codes");
constexpr uint32_t kOffTmemSlot = kOffBars + kNumBars * 8;
constexpr uint32_t kSmemUsed = kOffTmemSlot + 16;
constexpr uint32_t kSmemAlloc = kSmemUsed + 1024;  // room to align the base up to 1024
static_assert(kSmemAlloc <= 227 * 1024, "dynamic shared memory of one CTA on sm_103a");

constexpr uint32_t kIdescQK = ptx::idesc_bf16_f32(128, 128, false, false);
constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(128, 256, false, true);
constexpr uint32_t kIdescQK2 = ptx::idesc_bf16_f32(256, 128, false, false);  // CTA pair
constexpr uint32_t kIdescPV2 = ptx::idesc_bf16_f32(256, 256, false, true);   // CTA pair
constexpr uint32_t kIdescQK8 = ptx::idesc_e4m3_f32(128, 128);                 // FP8 QK^T
constexpr uint32_t kIdescQK82 = ptx::idesc_e4m3_f32(256, 128);                // FP8, pair
constexpr uint32_t kIdescPV8 = ptx::idesc_e4m3_f32(128, 256);                 // FP8 PV
constexpr uint32_t kIdescPV82 = ptx::idesc_e4m3_f32(256, 256);                // FP8 PV, pair

constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kRescaleThreshold = 8.0f;  // log2 units: p <= 2^8 between rescales
// Quantised PV: P is stored as the E4M3 code of 2^6 * p with the running maximum
// at most 2 below the row's maximum so far (p <= 4): 2^6 * p <= 256 < 448, and
// probabilities down to 2^-12 of the maximum stay in E4M3's normal range.
constexpr float kRescaleThresholdPv = 2.0f;
constexpr float kPScaleLog2Pv = 6.0f;
constexpr float kLn2 = 0.693147180559945309f;

__device__ int g_status_word = 0;

// Bounds-checked build (compiled with -DGQA_CHECK_BOUNDS, libgqa_prefill_checked.so):
// every global store of the epilogue and every read and write of the merge pass
// checks its row against the buffer's extent first; a row outside records
// GQA_ERR_BOUNDS in the status word and the access is skipped. (No device assert,
// no trap: the substitute for a memory checker, which this kernel's tests run under.)
#ifdef GQA_CHECK_BOUNDS
constexpr bool kCheckBounds = true;
#else
constexpr bool kCheckBounds = false;
#endif
__device__ __forceinline__ bool row_ok(long long r, long long rows, int* status) {
  if (!kCheckBounds || (r >= 0 && r < rows)) return true;
  atomicExch(status, static_cast<int>(GQA_ERR_BOUNDS));
  return false;
}

// Bounded wait for the phase of `bar` with the given parity.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const FwdParams& p) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t spin = 1;; ++spin) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((spin & 31u) == 0 && ptx::globaltimer_ns() - t0 > p.timeout_ns) {
      atomicExch(p.status, static_cast<int>(GQA_ERR_DEVICE_TIMEOUT));
      return false;
    }
  }
}

// wait_bar for a thread off the critical path (the paged kernel's two TMA
// producers): it sleeps in the barrier until the phase completes (or 20 us
// pass, then checks the time-out) instead of polling, leaving the issue slots
// of its scheduler to the softmax warp that shares it (polling cost the pair
// kernel ~3 % with two producer warps).
__device__ __forceinline__ bool wait_bar_idle(uint32_t bar, uint32_t parity, const FwdParams& p) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (;;) {
    if (ptx::mbar_try_wait_suspend(bar, parity, 20000u)) return true;
    if (ptx::globaltimer_ns() - t0 > p.timeout_ns) {
      atomicExch(p.status, static_cast<int>(GQA_ERR_DEVICE_TIMEOUT));
      return false;
    }
  }
}

// The V rows of the tile holding key kv_len-1 that lie past kv_len may hold
// anything: in a paged cache, the last page's unused slots; in a dense batch, the
// next sequence's values. Their P is exactly 0, but 0 * NaN is not, so they are
// zeroed before the PV reads the stage. The producer loads that tile's V in
// 16-key pieces and pieces that start past kv_len read TMA zero fill, so only
// keys [kv_len, next multiple of 16) remain. `base`: the stage (this CTA's
// shared::cta address, or the peer's shared::cluster address when `remote`),
// holding keys key0 .. key0+rows-1 of the tile (kr: its first key past kv_len);
// key r, chunk c at (r / 8) * sbo + c * lbo + (r % 8) * 128 (the stage layout's
// strides; a 128-byte row stays in place under the 128-byte swizzle). Out of
// line (rare: once per item that reaches the last KV tile) so the PV thread's
// loop stays small.
__device__ __noinline__ void zero_v_tail(uint32_t base, int nch, uint32_t sbo, uint32_t lbo,
                                         int key0, int rows, int kr, bool remote) {
  const int r_begin = max(kr, key0) - key0;
  const int r_end = min((kr + 15) & ~15, key0 + rows) - key0;
  for (int r = r_begin; r < r_end; ++r)
    for (int c = 0; c < nch; ++c)
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t a = base + (r >> 3) * sbo + c * lbo + (r & 7) * 128 + u * 16;
        if (remote) ptx::st_cluster_zero16(a); else ptx::st_shared_zero16(a);
      }
}

// Dense batch: the V box of the tile holding key kv_len-1 of a sequence, as
// 16-key pieces of one 64-column chunk each (4-D map, box (64, 16, 1, 1)):
// pieces that start past the sequence's kv_len keys read row oob_row, past the
// tensor (TMA zero fill), so that no value of the next sequence lands in the
// stage but the < 16 rows zero_v_tail clears. `r0`: first key of the box within
// the sequence; the stage is chunk-major with `rows` keys per chunk.
template <bool kPair>
__device__ __noinline__ void issue_dense_v_pieces(const CUtensorMap* map16, uint32_t dst,
                                                  uint32_t bar, int kv_start, int kv_len,
                                                  int oob_row, int r0, int rows, int nch,
                                                  int chunk0, int g, uint64_t pol) {
  for (int c = 0; c < nch; ++c)
    for (int i = 0; i < rows / 16; ++i) {
      const int key = r0 + 16 * i;
      const int row = key < kv_len ? kv_start + key : oob_row;
      const uint32_t d = dst + c * rows * 128 + i * 16 * 128;
      if constexpr (kPair) ptx::tma_load_4d_pair(d, map16, bar, 0, row, g, chunk0 + c, pol);
      else ptx::tma_load_4d(d, map16, bar, 0, row, g, chunk0 + c, pol);
    }
}

// Paged K/V: a box that crosses pages (or the V box of the tile holding key
// kv_len-1) goes as pieces (gqa_paged.h's map_paged_run), one 5-D copy per
// piece covering all `nch` chunks (paged stage layout, see the kernel). `bar`:
// the barrier the copies complete on (the pair leader's, mapped, for pairs).
// Inlined: as a call it cost the producer ~1,500 more cycles per box (per-tile
// clock traces, page 64).
template <bool kPair>
__device__ __forceinline__ void issue_paged_pieces(const PagedRun& run, const CUtensorMap* sub_map,
                                                   uint32_t dst, uint32_t bar, int nch, int chunk0,
                                                   int g, uint64_t pol) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {  // unrolled: run.row stays in registers
    if (i >= run.n) break;
    // Piece i is 8-key groups [i*sub/8, (i+1)*sub/8) of the stage: contiguous.
    const uint32_t d = dst + i * run.sub * nch * 128;
    if constexpr (kPair) ptx::tma_load_5d_pair(d, sub_map, bar, 0, 0, chunk0, run.row[i] / 8, g, pol);
    else ptx::tma_load_5d(d, sub_map, bar, 0, 0, chunk0, run.row[i] / 8, g, pol);
  }
}

// Paged FP8 K: the 128 key scales of tile key r0.. of head g into a ring slot.
// The scales sit in head-major rows beside the cache rows, so the same page
// mapping applies: one run inside a page, else pieces of sub_rows keys. Each is
// a 1-D bulk copy (16-byte alignment; a tensor copy would need its shared
// destination on 128 bytes, which 16-key pieces are not). Pieces past the
// cache or on a bad table entry are not copied but zeroed, and only the bytes
// actually copied are expected on `bar`; this thread's arrive (after the
// zeroing) is the slot's one arrival. Inlined, like issue_paged_pieces.
__device__ __forceinline__ void issue_paged_scales(const PagedGeom pgeo, const int* table,
                                                   int* status, const float* scale_row,
                                                   uint32_t dst, uint32_t bar, int r0,
                                                   uint64_t pol) {
  PagedRun run;
  map_paged_run(pgeo, r0, kBlockN, false, [&](int pg) { return __ldg(table + pg); }, run);
  if (run.bad) atomicExch(status, static_cast<int>(GQA_ERR_PAGE_TABLE));
  const int n = run.n == 0 ? 1 : run.n;
  const int keys = run.n == 0 ? kBlockN : run.sub;
  uint32_t bytes = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {  // unrolled: run.row stays in registers
    if (i >= n) break;
    if (run.row[i] < pgeo.oob_row) {
      bytes += keys * 4;
    } else {
      for (int c = 0; c < keys; c += 4) ptx::st_shared_zero16(dst + (i * keys + c) * 4);
    }
  }
  ptx::mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (i >= n) break;
    if (run.row[i] < pgeo.oob_row)
      ptx::bulk_load(dst + i * keys * 4, scale_row + run.row[i], keys * 4, bar, pol);
  }
}

// kPair = false: one CTA per work item (21 tokens x 6 heads = 126 MMA rows).
// kPair = true: a cluster of two CTAs per work item (42 tokens); CTA r holds
// tokens 21r .. 21r+20 (its own 128 MMA rows), the pair's leader (r = 0)
// issues cta_group::2 MMAs with M = 256, and each CTA loads half of every K
// tile (64 keys) and half of every V tile (128 of the 256 columns), so each
// SM streams and re-reads half the B operands of the one-CTA kernel. TMA
// copies of both CTAs complete on the leader's barriers; MMA completions are
// multicast to both CTAs; the peer's softmax warps arrive on the leader's
// barriers remotely.
//
// kFp8 = 2: also quantised PV (the same report's final submission): V arrives as
// E4M3 codes transposed per channel ([head][channel][key], one scale per
// channel), P is rounded to E4M3 as 2^6 * p, O += P V is a kind::f8f6f4 MMA with
// P from tensor memory and V K-major, and the epilogue multiplies column c of O
// by channel c's scale. Dense K/V, one sequence.
//
// kFp8 = 1: quantised QK^T (gfx936 DCU上实现INT8 QK MMAC, §1): Q and K are E4M3
// codes with one FP32 scale per query (token, head) and per key (token, KV
// head); S = Q_q K_q^T is a kind::f8f6f4 MMA, and every score is restored as
// S * s_q * s_k * scale before the softmax. PV stays BF16.
// Tensor-memory load / store of one thread's N consecutive 32-bit columns.
template <int N>
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, uint32_t (&r)[N]) {
  static_assert(N == 64 || N == 128, "64 or 128 columns");
  if constexpr (N == 64) ptx::tmem_ld_x64(taddr, r); else ptx::tmem_ld_x128(taddr, r);
}
template <int N>
__device__ __forceinline__ void tmem_st_n(uint32_t taddr, const uint32_t (&r)[N]) {
  static_assert(N == 16 || N == 32 || N == 64, "16, 32 or 64 columns");
  if constexpr (N == 16) ptx::tmem_st_x16(taddr, r);
  else if constexpr (N == 32) ptx::tmem_st_x32(taddr, r);
  else ptx::tmem_st_x64(taddr, r);
}

// Transpose of an 8 x 8 matrix of 16-byte quads held by a group of 8 lanes
// (aligned: lanes 8i .. 8i+7), lane j holding row j: afterwards lane j holds
// column j, e[s] = old e[j] of lane s. Three butterfly stages; in stage m the
// lanes whose bit m is set trade their quads i (bit m clear) for their
// partner's quads i | m. Used by the epilogue so that each store instruction
// of a group writes 128 contiguous bytes of one output row.
__device__ __forceinline__ void transpose8_quads(uint4 (&e)[8], int j) {
#pragma unroll
  for (int m = 4; m >= 1; m >>= 1) {
    const bool up = (j & m) != 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i & m) continue;
      const uint4 send = up ? e[i] : e[i | m];
      uint4 recv;
      recv.x = __shfl_xor_sync(0xffffffffu, send.x, m);
      recv.y = __shfl_xor_sync(0xffffffffu, send.y, m);
      recv.z = __shfl_xor_sync(0xffffffffu, send.z, m);
      recv.w = __shfl_xor_sync(0xffffffffu, send.w, m);
      if (up) e[i] = recv;
      else e[i | m] = recv;
    }
  }
}

// kKv: 0 dense K/V of one sequence; 1 paged K/V; 2 dense K/V of a batch of
// sequences packed end to end (the V box of a sequence's last tile goes in 16-key
// pieces so that the next sequence's values never reach it).
template <bool kPair, int kKv, int kFp8>
__global__ void __launch_bounds__(fwd_threads(kFp8, kKv), 1)
    gqa_attn_fwd_sm103_kernel(const __grid_constant__ FwdParams p) {
  constexpr bool kPaged = kKv == 1;
  constexpr bool kDenseBatch = kKv == 2;
  static_assert(kFp8 != 2 || kKv == 0, "quantised PV reads the dense V of one sequence");
  constexpr bool kFp8Pv = kFp8 == 2;
  // Warp roles: softmax warps 0 .. kSmWarps-1, then the TMA warp, the two MMA
  // warps and, for paged K/V, the V TMA warp.
  // With 8 softmax warps, warps q and q + 4 share the MMA rows (tensor-memory
  // lanes) 32q .. 32q+31 and take keys 0-63 and 64-127 of every tile.
  constexpr int kSmWarps = fwd_softmax_warps(kFp8);
  constexpr int kTmaWarp = kSmWarps;
  constexpr int kMmaWarp = kSmWarps + 1;  // QK^T issuer; allocates tensor memory
  constexpr int kPvWarp = kSmWarps + 2;   // PV issuer
  constexpr bool kSplitProducer = fwd_split_producer(kKv);
  constexpr int kTmaVWarp = kSmWarps + 3; // paged K/V: V producer (kTmaWarp: Q and K)
  constexpr int kHalves = kSmWarps / 4;  // softmax threads per MMA row
  constexpr int kCols = 128 / kHalves;   // scores of a tile per softmax thread
  static_assert(kHalves == 1 || kFp8 == 2, "the split softmax uses the exchange slots of the FP8 layout");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* const smem = smem_raw + (base - raw_base);
  const uint32_t q_smem = base + kOffQ;
  const uint32_t stage_smem = base + kOffStages;
  auto bar = [&](uint32_t id) { return base + kOffBars + 8u * id; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmemSlot);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = kPair ? ptx::cluster_ctarank() : 0u;  // position in the pair
  const bool leader = rank == 0;
  // Barriers the leader's MMA threads wait on, as seen from this CTA.
  auto lbar = [&](uint32_t id) { return kPair ? ptx::map_to_cta(bar(id), 0) : bar(id); };
  auto arrive_leader = [&](uint32_t id) {
    if constexpr (kPair) ptx::mbar_arrive_cluster(lbar(id)); else ptx::mbar_arrive(bar(id));
  };
  auto commit = [&](uint32_t id) {
    if constexpr (kPair) ptx::tc_commit_pair(bar(id)); else ptx::tc_commit(bar(id));
  };
  constexpr uint32_t kConsumers = (kPair ? 2 : 1) * kSmWarps * 32;  // softmax threads per item
  // Shared-memory layout of a K or V stage (its keys x nch 64-column chunks,
  // 128-byte rows, 128B swizzle). Dense K/V: chunk-major, each chunk's keys
  // contiguous (one 4-D copy per stage). Paged K/V: 8-key groups outermost with
  // the chunks inside each group, so that a piece of whole groups — what a
  // paged box that crosses a page is cut into — is contiguous and one 5-D
  // copy. Both are uniform strides for the MMA descriptors: K rows 8 apart at
  // kSboK, next chunk at kChunkK; V next chunk at kLboV, next 8 keys at kSboV.
  // Q and K rows hold 64 BF16 or 128 FP8 values per 128-byte chunk.
  constexpr int kQChunks = kFp8 ? 2 : 4;
  constexpr int kChunkElems = kFp8 ? 128 : 64;
  constexpr int kKStagesPerTile = (kFp8 || kPair) ? 1 : 2;
  constexpr int kVStagesPerTile = (kPair || kFp8Pv) ? 1 : 2;
  // The 5 stages form two rings, each filled in order by the producer and read in
  // order by one MMA thread: K stages 0 .. kStagesK-1 (QK^T thread), V stages
  // kStagesK .. 4 (PV thread). (With one ring read by both threads, a thread could
  // wait on a stage whose previous fill, for the other thread, was still in
  // flight, and take that stage's older phase for the one it waits for.)
  constexpr uint32_t kStagesK = kKStagesPerTile == 2 ? 3 : 2;  // 1.5 or 2 K tiles
  constexpr uint32_t kStagesV = kStages - kStagesK;
  static_assert(kStagesK >= kKStagesPerTile + 1 && kStagesV >= kVStagesPerTile,
                "each ring holds more than one tile's K, and at least one tile's V");
  constexpr uint32_t kNchK = kFp8 ? 2 : (kPair ? 4 : 2);  // chunks per K stage
  constexpr uint32_t kNchV = kPair ? 2 : 4;               // chunks per V stage
  constexpr uint32_t kRowsK = kPair ? 64 : 128;  // keys per K stage
  constexpr uint32_t kRowsV = kPair ? 128 : 64;  // keys per V stage
  constexpr uint32_t kChunkK = kPaged ? 1024u : kRowsK * 128u;
  constexpr uint32_t kSboK = kPaged ? kNchK * 1024u : 1024u;
  constexpr uint32_t kLboV = kPaged ? 1024u : kRowsV * 128u;
  constexpr uint32_t kSboV = kPaged ? kNchV * 1024u : 1024u;
  constexpr uint32_t kKStageBytes = kRowsK * kNchK * 128u;  // K bytes per stage per CTA
  // Quantised PV: a V tile is one stage of 128-byte rows of 128 key codes, one row
  // per channel (256, or this CTA's 128 in a pair): K-major, SBO = 8 rows.
  constexpr uint32_t kVStageBytesPv = kPair ? 16384u : 32768u;

  // The stream's next kernel (the split merge, or the caller's) may be
  // scheduled now; it waits for this grid to finish before touching memory.
  ptx::griddep_launch_dependents();

  // ---- set-up: barriers, idle Q rows, tensor memory -------------------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(bar(kBarFull + s), 1);
      ptx::mbar_init(bar(kBarEmpty + s), 1);
    }
    ptx::mbar_init(bar(kBarQFull), 1);
    ptx::mbar_init(bar(kBarQEmpty), 1);
    ptx::mbar_init(bar(kBarSFull), 1);
    ptx::mbar_init(bar(kBarSFree), kConsumers);
    ptx::mbar_init(bar(kBarPFull0), kConsumers);
    ptx::mbar_init(bar(kBarPFull1), kConsumers);
    ptx::mbar_init(bar(kBarPvDone0), 1);
    ptx::mbar_init(bar(kBarPvDone1), 1);
    ptx::mbar_init(bar(kBarOFree), kConsumers);
    ptx::mbar_init(bar(kBarDrain), 2);  // both MMA threads commit
    if constexpr (kFp8) {
      for (int i = 0; i < kScSlots; ++i) {
        ptx::mbar_init(bar(kBarScFull + i), 1);
        ptx::mbar_init(bar(kBarScEmpty + i), kSmWarps * 32);  // this CTA's softmax threads
      }
    }
    if constexpr (kHalves == 2)
      for (int i = 0; i < 4; ++i) ptx::mbar_init(bar(kBarXch + i), 2 * 32);
    ptx::fence_mbar_init();
  }
  if (warp < 4) {
    // Rows 126 and 127 of each Q chunk are never written by TMA: zero them once.
    for (int i = threadIdx.x; i < kQChunks * 2 * 128 / 16; i += 128) {
      const int chunk = i / 16, off = (i % 16) * 16;
      *reinterpret_cast<uint4*>(smem + kOffQ + chunk * kQChunkBytes + kQBoxBytes + off) =
          make_uint4(0, 0, 0, 0);
    }
    ptx::fence_proxy_async_smem();
  }
  if (warp == kMmaWarp) {
    if constexpr (kPair) {
      ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), kTmemCols);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if constexpr (kPair) ptx::cluster_sync();  // both CTAs' barriers exist before any remote use
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Everything above touched only this CTA's own on-chip state; from here on
  // global memory is read and written, so the previous kernel of the stream
  // must have completed (programmatic dependent launch overlaps the set-up).
  ptx::griddep_wait();
  const int tpi = kPair ? 2 * kTokPerTile : kTokPerTile;  // tokens per work item
  const int n_workers = kPair ? static_cast<int>(gridDim.x) / 2 : static_cast<int>(gridDim.x);
  const int worker = kPair ? static_cast<int>(blockIdx.x) / 2 : static_cast<int>(blockIdx.x);
  const Schedule sched{p.head_items, p.tail_splits, p.n_units, p.n_tail};
  PieceIter pieces;  // this CTA's (pair's) work, in order; each role walks its own copy
  pieces.init(&p.batch, p.tail.v, sched, n_workers, worker);
  // KV tile holding key kv_len-1 of a sequence when it is partial (else -1).
  auto v_fix_tile = [](const SeqGeo& sq) { return sq.kv_len % kBlockN ? (sq.kv_len - 1) / kBlockN : -1; };

  if (warp == kTmaWarp || (kSplitProducer && warp == kTmaVWarp)) {
    // ======================= TMA producers =====================================
    // Dense K/V: one thread, lane 0 of warp kTmaWarp, loads Q and fills both
    // rings in the order K0, K1, V0, K2, V1, ... Paged K/V: two threads each fill
    // one ring in tile order, lane 0 of warp kTmaWarp Q, the K ring and (FP8)
    // the key scales, lane 0 of warp kTmaVWarp the V ring. Issuing a copy
    // occupies the thread for a few hundred cycles, and a paged box adds its
    // block-table reads, or, where it crosses pages, one copy per piece: one
    // thread for both rings was the bottleneck (page 64: the pair kernel took
    // twice as long as on dense K/V; page 784: 1.3x; the one-CTA kernel, whose V
    // ring holds one tile, 1.17x even at page 1024). On dense K/V the second
    // thread gains nothing and its warp cost ~2 % (it shares a scheduler with a
    // softmax warp), so there one thread stays.
    constexpr bool split = kSplitProducer;
    if (lane == 0) {
      auto produce = [&](auto do_k_c, auto do_v_c) {
        constexpr bool do_k = decltype(do_k_c)::value;  // Q, the K ring, key scales
        constexpr bool do_v = decltype(do_v_c)::value;  // the V ring
        if constexpr (do_k) {
          ptx::prefetch_tmap(&p.tmap_q);
          ptx::prefetch_tmap(&p.tmap_k);
          if constexpr (kFp8) ptx::prefetch_tmap(&p.tmap_ks);
          if constexpr (kPaged) ptx::prefetch_tmap(&p.tmap_k_sub);
        }
        if constexpr (do_v) {
          ptx::prefetch_tmap(&p.tmap_v);
          if constexpr (kPaged) {
            ptx::prefetch_tmap(&p.tmap_v_sub);
            ptx::prefetch_tmap(&p.tmap_v16);
          }
        }
        // K/V tiles stay in L2 for the other items that read them; in decode-sized
        // calls no other item does, and they go first.
        const uint64_t pol_kv = p.kv_read_once ? ptx::policy_evict_first() : ptx::policy_evict_last();
        const uint64_t pol_q = ptx::policy_evict_first();
        // This thread's stages: ring0 .. ring_end-1 (absolute indices).
        constexpr uint32_t ring0 = do_k ? 0u : kStagesK;
        constexpr uint32_t ring_end = do_v ? static_cast<uint32_t>(kStages) : kStagesK;
        uint32_t kst = 0, kph = 0, vst = kStagesK, vph = 0;  // next stage and phase of each ring
        uint32_t issued_mask = 0, issued_parity = 0;  // per stage: a load issued / its phase
        uint32_t sc_count = 0, sc_issued_mask = 0, sc_issued_parity = 0;  // FP8 key-scale ring
        bool q_issued = false;
        uint32_t q_parity = 0;
        bool ok = true;
        auto load = [&](uint32_t dst, const CUtensorMap* map, uint32_t id, int c0, int c1, int c2,
                        uint64_t pol) {
          if constexpr (kPair) ptx::tma_load_3d_pair(dst, map, lbar(id), c0, c1, c2, pol);
          else ptx::tma_load_3d(dst, map, bar(id), c0, c1, c2, pol);
        };
        // A whole K/V box: 4-D (64 d, key, head, chunk) dense, 5-D (64 d, key % 8,
        // chunk, key / 8, head) paged; both with the stage layout described above.
        auto load_box = [&](uint32_t dst, const CUtensorMap* map, uint32_t id, int row, int g,
                            int chunk0) {
          if constexpr (kPaged) {
            if constexpr (kPair) ptx::tma_load_5d_pair(dst, map, lbar(id), 0, 0, chunk0, row / 8, g, pol_kv);
            else ptx::tma_load_5d(dst, map, bar(id), 0, 0, chunk0, row / 8, g, pol_kv);
          } else {
            if constexpr (kPair) ptx::tma_load_4d_pair(dst, map, lbar(id), 0, row, g, chunk0, pol_kv);
            else ptx::tma_load_4d(dst, map, bar(id), 0, row, g, chunk0, pol_kv);
          }
        };
        // Block-table entries (paged K/V): the K and V streams each keep the last
        // one they read, reset when an item of another sequence starts.
        [[maybe_unused]] int cached_pg[2] = {-1, -1}, cached_entry[2] = {0, 0};
        // One K tile is two 32 KB stages (d halves) in the one-CTA kernel and one
        // stage (this CTA's 64 keys) in a pair; likewise for V (key halves / this
        // CTA's 128 columns). A whole box is one copy; a paged box that crosses a
        // page is one copy per piece.
        auto next_tile = [&](const SeqGeo& sq, int n, auto is_k_c, int g) -> bool {
          constexpr bool is_k = decltype(is_k_c)::value;
          const bool v_fix = (kPaged || kDenseBatch) && !is_k && n == v_fix_tile(sq);
          const CUtensorMap* full = is_k ? &p.tmap_k : &p.tmap_v;
          [[maybe_unused]] const CUtensorMap* sub_map =
              is_k ? &p.tmap_k_sub : (v_fix ? &p.tmap_v16 : &p.tmap_v_sub);
          constexpr int halves = is_k ? kKStagesPerTile : kVStagesPerTile;
#pragma unroll 1
          for (int half = 0; half < halves; ++half) {
            uint32_t& st = is_k ? kst : vst;
            uint32_t& phase = is_k ? kph : vph;
            // The box's geometry and its block-table entries do not depend on the
            // stage: they are worked out (and the reads issued) before the wait for
            // a free stage, so that once one frees only the copies are left.
            // Box geometry: first key, keys per box, chunks and their stride in
            // shared memory, first chunk.
            int r0, rows, nb, chunk0;
            if constexpr (kPair) {
              r0 = n * kBlockN + (is_k ? 64 * static_cast<int>(rank) : 0);
              rows = is_k ? 64 : 128;
              nb = is_k ? static_cast<int>(kNchK) : 2;
              chunk0 = is_k ? 0 : 2 * static_cast<int>(rank);
            } else {
              r0 = n * kBlockN + (is_k ? 0 : 64 * half);
              rows = is_k ? 128 : 64;
              nb = is_k ? static_cast<int>(kNchK) : 4;
              chunk0 = is_k ? static_cast<int>(kNchK) * half : 0;
            }
            int row = sq.kv_start + r0;  // dense K/V: the box is the keys themselves
            bool whole = true;
            [[maybe_unused]] PagedRun run;  // the pieces of a paged box that crosses pages
            if constexpr (kPaged) {
              const int* table = p.block_table + static_cast<size_t>(sq.src) * p.bt_stride;
              constexpr int sid = is_k ? 0 : 1;
              auto read = [&](int pg) -> int {
                if (pg != cached_pg[sid]) {
                  cached_entry[sid] = __ldg(table + pg);
                  cached_pg[sid] = pg;
                }
                return cached_entry[sid];
              };
              const PagedGeom pgeo{sq.kv_len, p.page_size, p.num_pages, p.sub_rows, p.oob_row};
              bool bad = false;
              whole = paged_whole_box(pgeo, r0, rows, v_fix, read, &row, &bad);
              if (!whole) {
                map_paged_run(pgeo, r0, rows, v_fix, [&](int pg) { return __ldg(table + pg); }, run);
                bad = run.bad;
              }
              if (bad) atomicExch(p.status, static_cast<int>(GQA_ERR_PAGE_TABLE));
            }
            if (!(split ? wait_bar_idle(bar(kBarEmpty + st), phase ^ 1u, p)
                        : wait_bar(bar(kBarEmpty + st), phase ^ 1u, p)))
              return false;
            const uint32_t dst = stage_smem + st * kStageBytes;
            const uint32_t bytes = is_k ? kKStageBytes : (kFp8Pv ? kVStageBytesPv : kStageBytes);
            if (leader) ptx::mbar_arrive_expect_tx(bar(kBarFull + st), (kPair ? 2 : 1) * bytes);
            if constexpr (kPaged) {
              if (!whole)
                issue_paged_pieces<kPair>(run, sub_map, dst,
                                          kPair ? lbar(kBarFull + st) : bar(kBarFull + st), nb,
                                          chunk0, g, pol_kv);
            }
            if (kFp8Pv && !is_k)  // one box (128 keys, 256 or 128 channels, head g)
              load(dst, &p.tmap_v, kBarFull + st, sq.kv_start + n * kBlockN,
                   kPair ? 128 * static_cast<int>(rank) : 0, g, pol_kv);
            else if (kDenseBatch && v_fix)
              issue_dense_v_pieces<kPair>(&p.tmap_v16, dst, kPair ? lbar(kBarFull + st) : bar(kBarFull + st),
                                          sq.kv_start, sq.kv_len, p.oob_row, r0, rows, nb, chunk0, g,
                                          pol_kv);
            else if (whole)
              load_box(dst, full, kBarFull + st, row, g, chunk0);
            issued_mask |= 1u << st;
            issued_parity = (issued_parity & ~(1u << st)) | (phase << st);
            if (is_k) {
              if (++st == kStagesK) {
                st = 0;
                phase ^= 1u;
              }
            } else if (++st == kStages) {
              st = kStagesK;
              phase ^= 1u;
            }
          }
          if constexpr (kFp8 && is_k) {
            // The tile's 128 key scales of group g, for this CTA's softmax warps
            // (each CTA of a pair loads its own copy on its own barrier).
            const uint32_t slot = sc_count % kScSlots, use = sc_count / kScSlots;
            if (use > 0 && !wait_bar(bar(kBarScEmpty + slot), (use - 1) & 1u, p)) return false;
            const uint32_t sdst = base + kOffScales + slot * kScSlotBytes;
            if constexpr (kPaged) {  // the scales sit beside the cache rows: same page mapping
              const int* table = p.block_table + static_cast<size_t>(sq.src) * p.bt_stride;
              const PagedGeom pgeo{sq.kv_len, p.page_size, p.num_pages, p.sub_rows, p.oob_row};
              issue_paged_scales(pgeo, table, p.status,
                                 p.k_scale + static_cast<size_t>(g) * p.k_scale_stride, sdst,
                                 bar(kBarScFull + slot), n * kBlockN, pol_kv);
            } else {
              ptx::mbar_arrive_expect_tx(bar(kBarScFull + slot), kScSlotBytes);
              ptx::tma_load_2d(sdst, &p.tmap_ks, bar(kBarScFull + slot),
                               sq.ks_start + n * kBlockN, g, pol_kv);  // x: a multiple of 4
            }
            sc_issued_mask |= 1u << slot;
            sc_issued_parity = (sc_issued_parity & ~(1u << slot)) | ((use & 1u) << slot);
            ++sc_count;
          }
          return true;
        };
        int k = 0, last_seq = -1;
        Piece w;
        while (ok && pieces.next(w)) {
          const SeqGeo& sq = p.batch.seq[w.seq];
          if constexpr (kPaged) {
            if (w.seq != last_seq) cached_pg[0] = cached_pg[1] = -1;
          }
          last_seq = w.seq;
          if constexpr (do_k) {
            if (k > 0 && !(ok = wait_bar(bar(kBarQEmpty), (k - 1) & 1, p))) break;
            if (!(p.withhold_q && k == 0)) {
              if (leader)
                ptx::mbar_arrive_expect_tx(bar(kBarQFull), (kPair ? 2 : 1) * kQChunks * kQBoxBytes);
              for (int c = 0; c < kQChunks; ++c)
                load(q_smem + c * kQChunkBytes, &p.tmap_q, kBarQFull, kChunkElems * c, kGroup * w.g,
                     sq.q_start + tpi * w.qt + kTokPerTile * static_cast<int>(rank), pol_q);
              q_issued = true;
              q_parity = k & 1;
            }
          }
          if constexpr (do_k && do_v) {
            // K0, K1, V0, K2, V1, ..., V(nt-1)
            const int nt = w.n1 - w.n0;
            for (int j = 0; j < nt && ok; ++j) {
              ok = next_tile(sq, w.n0 + j, BoolC<true>{}, w.g);
              if (ok && j >= 1) ok = next_tile(sq, w.n0 + j - 1, BoolC<false>{}, w.g);
            }
            if (ok) ok = next_tile(sq, w.n1 - 1, BoolC<false>{}, w.g);
          } else {
            for (int n = w.n0; n < w.n1 && ok; ++n) ok = next_tile(sq, n, BoolC<do_k>{}, w.g);
          }
          ++k;
        }
        // Every copy issued must have landed before the CTA exits. On the normal
        // path the MMA threads already waited for all of them (these return at
        // once); after a time-out they may still be in flight. In a pair all
        // copies complete on the leader's barriers, so the leader drains for both.
        if (leader) {
          for (uint32_t s = ring0; s < ring_end; ++s)
            if (issued_mask & (1u << s)) wait_bar(bar(kBarFull + s), (issued_parity >> s) & 1u, p);
          if (q_issued) wait_bar(bar(kBarQFull), q_parity, p);
        }
        if constexpr (kFp8 && do_k) {  // key scales complete on each CTA's own barriers
          for (int s = 0; s < kScSlots; ++s)
            if (sc_issued_mask & (1u << s))
              wait_bar(bar(kBarScFull + s), (sc_issued_parity >> s) & 1u, p);
        }
      };
      if constexpr (!split) produce(BoolC<true>{}, BoolC<true>{});
      else if (warp == kTmaWarp) produce(BoolC<true>{}, BoolC<false>{});
      else produce(BoolC<false>{}, BoolC<true>{});
    }
    __syncwarp();
  } else if (warp == kMmaWarp || warp == kPvWarp) {
    // ======================= MMA issuers (the pair's leader) ===================
    // Two threads issue the MMAs: lane 0 of warp kMmaWarp the QK^T groups (QK_j
    // once the softmax holds S_{j-1}), lane 0 of warp kPvWarp the PV groups (PV_j
    // once P_j is written). A thread's first shared-memory access after a run of
    // tcgen05.mma (its next barrier wait) stalls for ~250 cycles while the tensor
    // pipe holds only a couple of its MMAs; with one issuing thread every such
    // wait between two groups left the pipe idle (per-tile traces: ~2 x 230
    // cycles of a 2,580-cycle BF16 tile). With two, one thread's MMAs keep the
    // pipe fed while the other waits. Each thread reads its own ring of K or V
    // stages in order; a commit tracks the MMAs of the committing thread only.
    if (lane == 0 && leader) {
      const bool is_qk = warp == kMmaWarp;
      const uint64_t q_desc0 = ptx::smem_desc(q_smem, 16, 1024, ptx::kSwizzle128B);
      const uint64_t k_desc0 = ptx::smem_desc(stage_smem, 16, kSboK, ptx::kSwizzle128B);
      const uint64_t v_desc0 = ptx::smem_desc(stage_smem, kLboV, kSboV, ptx::kSwizzle128B);
      // This thread's ring: stage st (absolute index), phase.
      const uint32_t ring0 = is_qk ? 0u : kStagesK, ring_end = is_qk ? kStagesK : kStages;
      uint32_t st = ring0, phase = 0;
      auto next_stage = [&] {
        if (++st == ring_end) { st = ring0; phase ^= 1u; }
      };
      uint32_t tile = 0;  // KV tiles this CTA has processed (global tile index T)
      bool ok = true;
      int k = 0;
      Piece w;
      while (ok && pieces.next(w)) {
        const int nt = w.n1 - w.n0;
        // S = Q K_j^T over d = 256 in k-steps of 16. Descriptors are built once;
        // an offset below 256 KB only touches the 14-bit start-address field, so
        // stepping through a tile is one add.
        auto issue_qk = [&](int j) -> bool {
          const uint32_t T = tile + j;
          // K arrives as kKStagesPerTile stages of kNchK 128-byte chunks (one-CTA
          // BF16: two d halves; pairs and FP8: one stage); every MMA advances
          // 32 bytes along d (16 BF16 or 32 FP8 values). The first K stage is waited
          // for before s_free: it has usually landed long before, and the wait for
          // the softmax is then the last thing between S being free and the MMAs.
          if (!wait_bar(bar(kBarFull + st), phase, p)) return false;
          // S may be overwritten once the softmax holds tile T-1's scores in registers.
          if (T > 0 && !wait_bar(bar(kBarSFree), (T - 1) & 1u, p)) return false;
          ptx::tc_fence_after();
#pragma unroll
          for (int half = 0; half < kKStagesPerTile; ++half) {
            if (half > 0 && !wait_bar(bar(kBarFull + st), phase, p)) return false;
            ptx::tc_fence_after();
            const uint64_t kd = k_desc0 + ((st * kStageBytes) >> 4);
#pragma unroll
            for (int c = 0; c < static_cast<int>(kNchK); ++c) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t a =
                    q_desc0 + (((half * kNchK + c) * kQChunkBytes + 32 * kk) >> 4);
                const uint64_t bd = kd + ((c * kChunkK + 32 * kk) >> 4);
                const uint32_t acc = (half | c | kk) != 0;
                if constexpr (kFp8) {
                  if constexpr (kPair) ptx::mma_ss_f8_pair(tmem + kTmemS, a, bd, kIdescQK82, acc);
                  else ptx::mma_ss_f8(tmem + kTmemS, a, bd, kIdescQK8, acc);
                } else {
                  if constexpr (kPair) ptx::mma_ss_pair(tmem + kTmemS, a, bd, kIdescQK2, acc);
                  else ptx::mma_ss(tmem + kTmemS, a, bd, kIdescQK, acc);
                }
              }
            }
            commit(kBarEmpty + st);
            next_stage();
          }
          commit(kBarSFull);
          if (j == nt - 1) commit(kBarQEmpty);
          return true;
        };
        auto issue_pv = [&](int j) -> bool {
          const uint32_t T = tile + j;
          const uint32_t b = T & 1u;
          // The (first) V stage before P, for the same reason as K before s_free.
          if (!wait_bar(bar(kBarFull + st), phase, p)) return false;
          if (!wait_bar(bar(b ? kBarPFull1 : kBarPFull0), (T >> 1) & 1u, p)) return false;
          if (j == 0 && k > 0 && !wait_bar(bar(kBarOFree), (k - 1) & 1, p)) return false;
          ptx::tc_fence_after();
          // O += P_j V_j in k-steps of 16 keys, N = 256. V stages are MN-major:
          // LBO = next 64-wide d chunk (kLboV), SBO = next group of 8 keys (kSboV).
          const int vfix_tile = (kPaged || kDenseBatch) ? v_fix_tile(p.batch.seq[w.seq]) : -1;
          const bool v_fix = (kPaged || kDenseBatch) && w.n0 + j == vfix_tile;
          const int kr = p.batch.seq[w.seq].kv_len - vfix_tile * kBlockN;  // used when v_fix
          if constexpr (kFp8Pv) {
            // One stage: (this CTA's) channel rows of 128 key codes, K-major; P as E4M3
            // in tensor memory (4 codes per column: 8 columns per 32-key k-step).
            ptx::tc_fence_after();
            const uint64_t vd = k_desc0 + ((st * kStageBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t a_tmem = tmem + kTmemP + 64u * b + 8u * kk;
              if constexpr (kPair)
                ptx::mma_ts_f8_pair(tmem + kTmemO, a_tmem, vd + ((32 * kk) >> 4), kIdescPV82,
                                    (j | kk) != 0);
              else
                ptx::mma_ts_f8(tmem + kTmemO, a_tmem, vd + ((32 * kk) >> 4), kIdescPV8,
                               (j | kk) != 0);
            }
            commit(kBarEmpty + st);
            next_stage();
          } else if constexpr (kPair) {
            // One stage: 128 keys x this CTA's 2 chunks of 64 columns (waited for above).
            ptx::tc_fence_after();
            if (v_fix) {
              zero_v_tail(stage_smem + st * kStageBytes, kNchV, kSboV, kLboV, 0, kRowsV, kr, false);
              zero_v_tail(ptx::map_to_cta(stage_smem + st * kStageBytes, 1), kNchV, kSboV, kLboV, 0,
                          kRowsV, kr, true);
              ptx::fence_proxy_async_all();
            }
            const uint64_t vd = v_desc0 + ((st * kStageBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t bd = vd + ((2 * kSboV * kk) >> 4);  // 16 keys = two 8-key groups
              ptx::mma_ts_pair(tmem + kTmemO, tmem + kTmemP + 64u * b + 8u * kk, bd, kIdescPV2,
                               (j | kk) != 0);
            }
            commit(kBarEmpty + st);
            next_stage();
          } else {
            // Two stages (key halves), each 64 keys x 4 chunks of 64 d.
            for (int half = 0; half < 2; ++half) {
              if (half > 0 && !wait_bar(bar(kBarFull + st), phase, p)) return false;
              ptx::tc_fence_after();
              if (v_fix) {
                zero_v_tail(stage_smem + st * kStageBytes, kNchV, kSboV, kLboV, kRowsV * half, kRowsV,
                            kr, false);
                ptx::fence_proxy_async_all();
              }
              const uint64_t vd = v_desc0 + ((st * kStageBytes) >> 4);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t bd = vd + ((2 * kSboV * kk) >> 4);  // 16 keys = two 8-key groups
                const uint32_t a_tmem = tmem + kTmemP + 64u * b + 32u * half + 8u * kk;
                ptx::mma_ts(tmem + kTmemO, a_tmem, bd, kIdescPV, (j | half | kk) != 0);
              }
              commit(kBarEmpty + st);
              next_stage();
            }
          }
          commit(b ? kBarPvDone1 : kBarPvDone0);
          return true;
        };
        if (is_qk) {
          if (!(ok = wait_bar(bar(kBarQFull), k & 1, p))) break;
          ptx::tc_fence_after();
          for (int j = 0; j < nt && ok; ++j) ok = issue_qk(j);
        } else {
          for (int j = 0; j < nt && ok; ++j) ok = issue_pv(j);
        }
        tile += nt;
        ++k;
      }
      // Drain: every MMA issued above (both threads commit) has completed once
      // this barrier fires.
      commit(kBarDrain);
      wait_bar(bar(kBarDrain), 0, p);
    }
    __syncwarp();
  } else {
    // ======================= softmax + correction + epilogue (softmax warps) ===
    // Warp w owns MMA rows 32 (w % 4) .. +31 (a warp reaches only its quarter of
    // the tensor-memory lanes). With two threads per row, half hf = w / 4 takes
    // keys 64 hf .. 64 hf + 63 of every tile and columns 128 hf .. 128 hf + 127
    // of O; the two trade the row's tile maximum and, at the end, its sum.
    const int qw = warp & 3;
    const int hf = kHalves == 2 ? warp >> 2 : 0;
    const int row = qw * 32 + lane;  // MMA row == tensor-memory lane
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(qw * 32) << 16);
    const int kc0 = kCols * hf;                 // this thread's first key of a tile
    const int oc0 = (kHeadDim / kHalves) * hf;  // ... and first column of O
    // Trade of one value between the two threads of a row through shared memory:
    // slot xph & 1, then phase xph of the quarter's barrier (both threads trade in
    // the same order, so their counts agree; a slot is rewritten two trades later,
    // after the partner's next arrival, so its read of this one is done).
    uint32_t xph = 0;
    float* const xch = reinterpret_cast<float*>(smem + kOffXch);
    auto trade = [&](float v, float& other) -> bool {
      float* const slot = xch + (xph & 1u) * 256;
      slot[hf * 128 + row] = v;
      ptx::mbar_arrive(bar(kBarXch + qw));
      const bool good = __all_sync(0xffffffffu, wait_bar(bar(kBarXch + qw), xph & 1u, p));
      other = slot[(hf ^ 1) * 128 + row];
      ++xph;
      return good;
    };
    const int tl = row / kGroup;
    const int hj = row - tl * kGroup;
    const float sl2 = p.scale_log2;
    uint32_t tile = 0;
    int k = 0;
    bool ok = true;
    Piece w;
    while (ok && pieces.next(w)) {
      const int nt = w.n1 - w.n0;
      const SeqGeo& sq = p.batch.seq[w.seq];
      const int p0 = sq.kv_len - sq.q_len;   // position of the sequence's first new token
      const int tok0 = tpi * w.qt + kTokPerTile * static_cast<int>(rank);  // this CTA's first token
      const int tok = tok0 + tl;             // token within the sequence
      const bool valid = row < kTokPerTile * kGroup && tok < sq.q_len;
      const int pos = p0 + tok;              // last key this row may see
      const int tile_min_pos = p0 + tok0;    // smallest such key among this CTA's rows
      const size_t qrow = static_cast<size_t>(sq.q_start + tok) * kQHeads + kGroup * w.g + hj;
      // Score -> base-2 exponent factor: scale * log2(e), times the query's scale
      // for FP8 QK^T (the key's scale is applied per column below).
      float rowfac = sl2;
      if constexpr (kFp8) {
        // A query vector of zeros has scale 0 and codes 0: its scores are all 0. The
        // factor stays positive so that masked keys (-inf) stay -inf, not -inf * 0.
        if (valid) rowfac = sl2 * fmaxf(__ldg(p.q_scale + qrow), 1e-30f);
      }
      float m_ref = kNegInf;  // max used in the exponent (base-2, scaled)
      float l = 0.0f;         // running row sum of p
      for (int j = 0; j < nt; ++j) {
        const uint32_t T = tile + j;
        const uint32_t b = T & 1u;
        ok = __all_sync(0xffffffffu, wait_bar(bar(kBarSFull), T & 1u, p));
        if (!ok) break;
        ptx::tc_fence_after();
        uint32_t sr[kCols];
        tmem_ld_n(lane_addr + kTmemS + kc0, sr);  // includes tcgen05.wait::ld
        ptx::tc_fence_before();
        arrive_leader(kBarSFree);  // the next QK^T may overwrite S now
        float s[kCols];
#pragma unroll
        for (int c = 0; c < kCols; ++c) s[c] = __uint_as_float(sr[c]);
        if constexpr (kFp8) {
          // Restore each key's scale before the softmax (the report's §1: scales
          // change the relative probabilities, so they cannot wait until after).
          const uint32_t slot = T % kScSlots;
          ok = __all_sync(0xffffffffu, wait_bar(bar(kBarScFull + slot), (T / kScSlots) & 1u, p));
          if (!ok) break;
          const float4* ks =
              reinterpret_cast<const float4*>(smem + kOffScales + slot * kScSlotBytes) + kc0 / 4;
#pragma unroll
          for (int c = 0; c < kCols; c += 4) {
            const float4 k4 = ks[c / 4];
            float a0, a1, a2, a3;
            ptx::f32x2_split(ptx::mul_f32x2(ptx::f32x2(s[c], s[c + 1]), ptx::f32x2(k4.x, k4.y)), a0, a1);
            ptx::f32x2_split(ptx::mul_f32x2(ptx::f32x2(s[c + 2], s[c + 3]), ptx::f32x2(k4.z, k4.w)), a2, a3);
            s[c] = a0;
            s[c + 1] = a1;
            s[c + 2] = a2;
            s[c + 3] = a3;
          }
          ptx::mbar_arrive(bar(kBarScEmpty + slot));
        }
        const int key0 = (w.n0 + j) * kBlockN + kc0;  // key of s[0]
        if (key0 + kCols - 1 > tile_min_pos) {
          // Diagonal tile: keys after this row's position are masked out.
#pragma unroll
          for (int c = 0; c < kCols; ++c)
            if (key0 + c > pos) s[c] = kNegInf;
        }
        // Row maximum: four running maxima over s[], eight scores a step.
        float mx0 = kNegInf, mx1 = kNegInf, mx2 = kNegInf, mx3 = kNegInf;
#pragma unroll
        for (int c = 0; c < kCols; c += 8) {
          mx0 = ptx::fmax3(mx0, s[c], s[c + 1]);
          mx1 = ptx::fmax3(mx1, s[c + 2], s[c + 3]);
          mx2 = ptx::fmax3(mx2, s[c + 4], s[c + 5]);
          mx3 = ptx::fmax3(mx3, s[c + 6], s[c + 7]);
        }
        // (rowfac > 0: scaling each half's maximum gives the scaled row maximum exactly.)
        float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * rowfac;
        if constexpr (kHalves == 2) {
          float m_other;
          ok = trade(m_tile, m_other);
          if (!ok) break;
          m_tile = fmaxf(m_tile, m_other);
        }
        const float m_new = fmaxf(m_ref, m_tile);
        const bool need = m_new > m_ref + (kFp8Pv ? kRescaleThresholdPv : kRescaleThreshold);
        // O correction: P_j is computed against the new reference at once; O (which
        // must first hold PV_{j-1}) is rescaled after P_j is stored, just before
        // p_full, by which time PV_{j-1} has normally completed.
        bool rescale = false;
        float alpha = 1.0f;
        if (j == 0) {
          if (need) m_ref = m_new;  // O is overwritten by this unit's first PV
        } else if (__any_sync(0xffffffffu, need)) {
          alpha = need ? ptx::ex2_approx(m_ref - m_new) : 1.0f;
          if (need) m_ref = m_new;
          l *= alpha;
          rescale = true;
        }
        const float m_use = (m_ref == kNegInf) ? 0.0f : m_ref;
        // BF16 P: two values per tensor-memory column; E4M3 P (quantised PV): four.
        uint32_t pk[kFp8Pv ? kCols / 4 : kCols / 2];
        // p = 2^(s*scale*log2e - m): one packed FMA per pair, two ex2, one packed add.
        const uint64_t scale2 = ptx::f32x2(rowfac, rowfac);
        const float pofs = kFp8Pv ? kPScaleLog2Pv - m_use : -m_use;
        const uint64_t neg_m2 = ptx::f32x2(pofs, pofs);
        uint64_t sum2 = ptx::f32x2(0.0f, 0.0f);
#pragma unroll
        for (int c = 0; c < kCols / 2; ++c) {
          float x0, x1;
          ptx::f32x2_split(ptx::fma_f32x2(ptx::f32x2(s[2 * c], s[2 * c + 1]), scale2, neg_m2), x0, x1);
          const float e0 = ptx::ex2_approx(x0);
          const float e1 = ptx::ex2_approx(x1);
          sum2 = ptx::add_f32x2(sum2, ptx::f32x2(e0, e1));
          if constexpr (kFp8Pv) {
            const uint32_t h = ptx::cvt_e4m3x2(e0, e1);
            pk[c >> 1] = (c & 1) ? (pk[c >> 1] | (h << 16)) : h;
          } else {
            pk[c] = ptx::pack_bf16x2(e0, e1);
          }
        }
        float sum0, sum1;
        ptx::f32x2_split(sum2, sum0, sum1);
        l += sum0 + sum1;
        if (T >= 2) {
          // P[b] was last read by PV_{T-2}: it must have completed before P[b] is rewritten.
          ok = __all_sync(0xffffffffu, wait_bar(bar(b ? kBarPvDone1 : kBarPvDone0),
                                                ((T - 2) >> 1) & 1u, p));
          if (!ok) break;
          ptx::tc_fence_after();
        }
        // Key k of the tile sits in P column k / 2 (BF16) or k / 4 (E4M3).
        tmem_st_n(lane_addr + kTmemP + 64u * b + (kFp8Pv ? kc0 / 4 : kc0 / 2), pk);
        ptx::tmem_st_wait();
        if (rescale) {  // warp-uniform
          // O must hold PV_{j-1} (which read P[(T-1)&1], use (T-1)>>1) before it is rescaled.
          ok = __all_sync(0xffffffffu, wait_bar(bar((T - 1) & 1u ? kBarPvDone1 : kBarPvDone0),
                                                ((T - 1) >> 1) & 1u, p));
          if (!ok) break;
          ptx::tc_fence_after();
#pragma unroll 1
          for (int c = oc0; c < oc0 + kHeadDim / kHalves; c += 32) {
            uint32_t o[32];
            ptx::tmem_ld_x32(lane_addr + kTmemO + c, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            ptx::tmem_st_x32(lane_addr + kTmemO + c, o);
          }
          ptx::tmem_st_wait();
        }
        ptx::tc_fence_before();
        arrive_leader(b ? kBarPFull1 : kBarPFull0);
      }
      if (!ok) break;
      // ---- epilogue: O / l -> out (or the split partial), LSE ----------------
      const uint32_t T_last = tile + nt - 1;
      ok = __all_sync(0xffffffffu, wait_bar(bar(T_last & 1u ? kBarPvDone1 : kBarPvDone0),
                                            (T_last >> 1) & 1u, p));
      if (!ok) break;
      ptx::tc_fence_after();
      if constexpr (kHalves == 2) {  // the row sum: both halves' (IEEE + commutes: the same in both)
        float l_other;
        ok = trade(l, l_other);
        if (!ok) break;
        l += l_other;
      }
      const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;
      // (Quantised PV: l sums 2^6 p, so the scale's exponent comes off.)
      const float lse2 = l > 0.0f ? m_ref + __log2f(l) - (kFp8Pv ? kPScaleLog2Pv : 0.0f) : kNegInf;
      // Output column factor: 1/l, times the channel's V scale for quantised PV.
      auto col_factors = [&](int col0, float (&f)[32]) {
        if constexpr (kFp8Pv) {
          const float4* sv = reinterpret_cast<const float4*>(p.v_scale + kHeadDim * w.g + col0);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 x = __ldg(sv + i);
            f[4 * i] = x.x * inv_l; f[4 * i + 1] = x.y * inv_l;
            f[4 * i + 2] = x.z * inv_l; f[4 * i + 3] = x.w * inv_l;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) f[i] = inv_l;
        }
      };
      // Stores go out through groups of 8 lanes: after transpose8_quads each lane
      // of a group holds one 16-byte quad of each of the group's 8 rows, so every
      // store instruction writes 128 contiguous bytes of 4 rows instead of 16
      // bytes of 32 rows (the output rows are 512 bytes, partial rows 1 KB apart).
      const int gl = lane & 7;                    // lane within its group of 8
      const int grow0 = qw * 32 + (lane & ~7);  // MMA row of the group's lane 0
      auto group_row = [&](int s_, int& tok_s) -> bool {
        const int r = grow0 + s_;
        tok_s = tok0 + r / kGroup;
        return r < kTokPerTile * kGroup && tok_s < sq.q_len;
      };
      if (w.slot < 0) {
        size_t off[8];  // element offset of each group row in `out`
        uint32_t vmask = 0;
#pragma unroll
        for (int s_ = 0; s_ < 8; ++s_) {
          int tok_s;
          const bool v_ = group_row(s_, tok_s);
          const int hj_s = (grow0 + s_) % kGroup;
          off[s_] = (static_cast<size_t>(sq.q_start + tok_s) * kQHeads + kGroup * w.g + hj_s) * kHeadDim;
          vmask |= (v_ ? 1u : 0u) << s_;
        }
#pragma unroll 1
        for (int c = oc0; c < oc0 + kHeadDim / kHalves; c += 64) {
          uint4 e[8];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t o[32];
            ptx::tmem_ld_x32(lane_addr + kTmemO + c + 32 * h, o);
            float f[32];
            col_factors(c + 32 * h, f);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const int i = 8 * q4;
              e[4 * h + q4] = make_uint4(
                  ptx::pack_bf16x2(__uint_as_float(o[i]) * f[i], __uint_as_float(o[i + 1]) * f[i + 1]),
                  ptx::pack_bf16x2(__uint_as_float(o[i + 2]) * f[i + 2], __uint_as_float(o[i + 3]) * f[i + 3]),
                  ptx::pack_bf16x2(__uint_as_float(o[i + 4]) * f[i + 4], __uint_as_float(o[i + 5]) * f[i + 5]),
                  ptx::pack_bf16x2(__uint_as_float(o[i + 6]) * f[i + 6], __uint_as_float(o[i + 7]) * f[i + 7]));
            }
          }
          transpose8_quads(e, gl);
#pragma unroll
          for (int s_ = 0; s_ < 8; ++s_)
            if ((vmask & (1u << s_)) &&
                row_ok(static_cast<long long>(off[s_] / kHeadDim), p.out_rows, p.status))
              *reinterpret_cast<uint4*>(p.out + off[s_] + c + 8 * gl) = e[s_];
        }
        if (hf == 0 && valid && p.lse != nullptr &&
            row_ok(static_cast<long long>(qrow), p.out_rows, p.status))
          p.lse[qrow] = lse2 * kLn2;
      } else {
        // A piece of a split item: normalised partial rows go to the piece's slot
        // (one 128-row block per CTA of the item).
        const size_t slot_row0 =
            (static_cast<size_t>(w.slot) * (kPair ? 2 : 1) + rank) * kRowsPerTile;
        uint32_t vmask = 0;
#pragma unroll
        for (int s_ = 0; s_ < 8; ++s_) {
          int tok_s;
          vmask |= (group_row(s_, tok_s) ? 1u : 0u) << s_;
        }
        float* base = p.part_o + (slot_row0 + grow0) * kHeadDim;
#pragma unroll 1
        for (int c = oc0; c < oc0 + kHeadDim / kHalves; c += 32) {
          uint32_t o[32];
          ptx::tmem_ld_x32(lane_addr + kTmemO + c, o);
          float f[32];
          col_factors(c, f);
          uint4 e[8];
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4)
            e[q4] = make_uint4(__float_as_uint(__uint_as_float(o[4 * q4]) * f[4 * q4]),
                               __float_as_uint(__uint_as_float(o[4 * q4 + 1]) * f[4 * q4 + 1]),
                               __float_as_uint(__uint_as_float(o[4 * q4 + 2]) * f[4 * q4 + 2]),
                               __float_as_uint(__uint_as_float(o[4 * q4 + 3]) * f[4 * q4 + 3]));
          transpose8_quads(e, gl);
#pragma unroll
          for (int s_ = 0; s_ < 8; ++s_)
            if ((vmask & (1u << s_)) &&
                row_ok(static_cast<long long>(slot_row0 + grow0 + s_), p.part_rows, p.status))
              *reinterpret_cast<uint4*>(base + static_cast<size_t>(s_) * kHeadDim + c + 4 * gl) = e[s_];
        }
        if (hf == 0 && valid && row_ok(static_cast<long long>(slot_row0 + row), p.part_rows, p.status))
          p.part_lse[slot_row0 + row] = lse2;
      }
      ptx::tc_fence_before();
      arrive_leader(kBarOFree);
      tile += nt;
      ++k;
    }
  }

  // ---- teardown ----------------------------------------------------------------
  // In a pair, neither CTA may leave (or free tensor memory) while the leader's
  // MMAs or the peer's remote arrivals can still touch it.
  ptx::tc_fence_before();
  __syncthreads();
  if constexpr (kPair) ptx::cluster_sync();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    if constexpr (kPair) ptx::tmem_dealloc_pair(tmem, kTmemCols);
    else ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// Combine the pieces of every split (tail) item: blocks (j, *) merge tail item
// j (item head_items + j), 8 rows each. Its n pieces are read in KV order from
// their slots (each slot holds one 128-row block per CTA of the item): uniform
// tail, piece s in slot j*S + s; balanced tail, the workers' slots that
// balanced_item_pieces / balanced_slot name (an item that no worker boundary
// cuts was written whole by the attention kernel: its blocks return at once).
// lse = log2 sum_s 2^{lse_s}, out = sum_s 2^{lse_s - lse} O_s. One warp per row,
// every lane holding 8 columns: the loads of the first 4 pieces' columns and of
// every piece's LSE (lane s: piece s) go out together, so a row of up to 4
// pieces costs one memory round trip (registers stay under 64, four blocks per
// SM); the warp reduces max and sum by shuffles
// and accumulates the pieces in order s = 0, 1, ... (deterministic). With one
// row per warp every row of the call is in flight at once.
constexpr int kMergeRowsPerBlock = 8;  // 8 warps x 1 row
constexpr int kMergeBatch = 4;         // pieces whose columns a lane loads at once

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Every piece's LSE of one row, read by the lanes of a warp (lane s: piece s, 32
// per pass): returns the row's maximum and, in *l0, the lane's LSE of pass 0.
template <typename RowOf>
__device__ __forceinline__ float row_lse_max(const float* part_lse, int n, int lane, RowOf prow,
                                             float* l0) {
  *l0 = lane < n ? __ldcg(part_lse + prow(lane)) : kNegInf;
  float mx = *l0;
  for (int s0 = 32; s0 < n; s0 += 32)
    if (s0 + lane < n) mx = fmaxf(mx, __ldcg(part_lse + prow(s0 + lane)));
  return warp_max(mx);
}

// Weight 2^{lse_s - m} of piece s (lane-uniform s): from lane s's LSE for s < 32.
template <typename RowOf>
__device__ __forceinline__ float piece_weight(const float* part_lse, int s, float l0, float m,
                                              RowOf prow) {
  const float l = s < 32 ? __shfl_sync(0xffffffffu, l0, s) : __ldcg(part_lse + prow(s));
  return ptx::ex2_approx(l - m);
}

__global__ void __launch_bounds__(256, 4) merge_tail_kernel(const __grid_constant__ MergeParams p) {
  ptx::griddep_wait();  // launched early (programmatic dependent launch): the pieces must be done
  const int j = blockIdx.x;  // tail item
  const bool balanced = p.tail_splits == 0;
  int n = p.tail_splits, x_lo = 0;
  if (balanced) {
    balanced_item_pieces(p.tail.v, p.tail_items, p.workers, j, x_lo, n);
    if (n < 2) return;  // not split: written by the attention kernel
  }
  int seq, qt, g;
  item_of(p.batch, p.head_items + j, seq, qt, g);
  const SeqGeo& sq = p.batch.seq[seq];
  const int cpi = p.ctas_per_item;
  const int lane = threadIdx.x & 31;
  const int rr = blockIdx.y * kMergeRowsPerBlock + static_cast<int>(threadIdx.x >> 5);
  if (rr >= cpi * kTokPerTile * kGroup) return;
  const int r = rr / (kTokPerTile * kGroup);    // CTA of the item
  const int row = rr % (kTokPerTile * kGroup);  // its MMA row
  const int tok = kTokPerTile * (cpi * qt + r) + row / kGroup;  // token within the sequence
  if (tok >= sq.q_len) return;
  // Partial row of piece s: its slot, CTA r, MMA row `row`.
  auto prow = [&](int s) {
    const int slot = balanced ? balanced_slot(p.tail.v, p.tail_items, p.workers, j, x_lo, s)
                              : j * n + s;
    return (static_cast<size_t>(slot) * cpi + r) * kRowsPerTile + row;
  };
  if constexpr (kCheckBounds) {  // every partial row this warp will read
    bool rows_ok = true;
    for (int s0 = 0; s0 < n; s0 += 32)
      if (s0 + lane < n) rows_ok &= row_ok(static_cast<long long>(prow(s0 + lane)), p.part_rows, p.status);
    if (!__all_sync(0xffffffffu, rows_ok)) return;
  }
  auto cols = [&](int s) {
    return reinterpret_cast<const float4*>(p.part_o + prow(s) * kHeadDim + 8 * lane);
  };
  float4 va[kMergeBatch], vb[kMergeBatch];
#pragma unroll
  for (int i = 0; i < kMergeBatch; ++i)
    if (i < n) {
      va[i] = __ldcg(cols(i));
      vb[i] = __ldcg(cols(i) + 1);
    }
  float l0;
  const float mx = row_lse_max(p.part_lse, n, lane, prow, &l0);
  const float m_use = (mx == kNegInf) ? 0.0f : mx;
  float wsum = warp_sum(lane < n ? ptx::ex2_approx(l0 - m_use) : 0.0f);
  for (int s0 = 32; s0 < n; s0 += 32)
    wsum += warp_sum(s0 + lane < n ? ptx::ex2_approx(__ldcg(p.part_lse + prow(s0 + lane)) - m_use)
                                   : 0.0f);
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int s0 = 0; s0 < n; s0 += kMergeBatch) {
    if (s0 > 0) {
#pragma unroll
      for (int i = 0; i < kMergeBatch; ++i)
        if (s0 + i < n) {
          va[i] = __ldcg(cols(s0 + i));
          vb[i] = __ldcg(cols(s0 + i) + 1);
        }
    }
#pragma unroll
    for (int i = 0; i < kMergeBatch; ++i) {
      if (s0 + i >= n) break;
      const float w = piece_weight(p.part_lse, s0 + i, l0, m_use, prow);
      acc[0] += w * va[i].x; acc[1] += w * va[i].y; acc[2] += w * va[i].z; acc[3] += w * va[i].w;
      acc[4] += w * vb[i].x; acc[5] += w * vb[i].y; acc[6] += w * vb[i].z; acc[7] += w * vb[i].w;
    }
  }
  const float inv = wsum > 0.0f ? 1.0f / wsum : 0.0f;
  uint4 o;
  o.x = ptx::pack_bf16x2(acc[0] * inv, acc[1] * inv);
  o.y = ptx::pack_bf16x2(acc[2] * inv, acc[3] * inv);
  o.z = ptx::pack_bf16x2(acc[4] * inv, acc[5] * inv);
  o.w = ptx::pack_bf16x2(acc[6] * inv, acc[7] * inv);
  const size_t orow = static_cast<size_t>(sq.q_start + tok) * kQHeads + kGroup * g + row % kGroup;
  if (!row_ok(static_cast<long long>(orow), p.out_rows, p.status)) return;
  *reinterpret_cast<uint4*>(p.out + orow * kHeadDim + 8 * lane) = o;
  if (lane == 0 && p.lse != nullptr)
    p.lse[orow] = wsum > 0.0f ? (m_use + __log2f(wsum)) * kLn2 : kNegInf;
}

// The same merge for calls whose items have many pieces (decode-sized chunks cut
// into 16 or more KV pieces, on the uniform or the balanced tail): one block per
// row, its 8 warps taking the pieces s = w, w + 8, ... (each warp loads its first
// 6 pieces' columns together with every piece's LSE, one round trip for up to
// 48 pieces), their weighted partial sums combined through shared memory in warp
// order (fixed order: deterministic). Blocks (j, r): tail item j, row r of the
// item's rows.
constexpr int kWideWarps = 8;
constexpr int kWideMergePieces = 16;  // items with this many pieces or more use it
constexpr int kWideBatch = 6;         // pieces per warp whose columns load at once

__global__ void __launch_bounds__(kWideWarps * 32)
    merge_wide_kernel(const __grid_constant__ MergeParams p) {
  __shared__ float part[kWideWarps][kHeadDim];
  __shared__ float part_w[kWideWarps];
  ptx::griddep_wait();
  const int j = blockIdx.x;
  const bool balanced = p.tail_splits == 0;
  int n = p.tail_splits, x_lo = 0;
  if (balanced) {
    balanced_item_pieces(p.tail.v, p.tail_items, p.workers, j, x_lo, n);
    if (n < 2) return;
  }
  int seq, qt, g;
  item_of(p.batch, p.head_items + j, seq, qt, g);
  const SeqGeo& sq = p.batch.seq[seq];
  const int cpi = p.ctas_per_item;
  const int rr = blockIdx.y;
  if (rr >= cpi * kTokPerTile * kGroup) return;
  const int r = rr / (kTokPerTile * kGroup);
  const int row = rr % (kTokPerTile * kGroup);
  const int tok = kTokPerTile * (cpi * qt + r) + row / kGroup;
  if (tok >= sq.q_len) return;  // the whole block leaves together
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto prow = [&](int s) {
    const int slot = balanced ? balanced_slot(p.tail.v, p.tail_items, p.workers, j, x_lo, s)
                              : j * n + s;
    return (static_cast<size_t>(slot) * cpi + r) * kRowsPerTile + row;
  };
  if constexpr (kCheckBounds) {
    bool rows_ok = true;
    for (int s = threadIdx.x; s < n; s += kWideWarps * 32)
      rows_ok &= row_ok(static_cast<long long>(prow(s)), p.part_rows, p.status);
    if (!__syncthreads_and(rows_ok)) return;
  }
  auto cols = [&](int s) {
    return reinterpret_cast<const float4*>(p.part_o + prow(s) * kHeadDim + 8 * lane);
  };
  float4 va[kWideBatch], vb[kWideBatch];
#pragma unroll
  for (int i = 0; i < kWideBatch; ++i) {
    const int s = warp + kWideWarps * i;
    if (s < n) {
      va[i] = __ldcg(cols(s));
      vb[i] = __ldcg(cols(s) + 1);
    }
  }
  // Every warp finds the row's maximum piece LSE itself (n loads across the lanes).
  float l0;
  const float mx = row_lse_max(p.part_lse, n, lane, prow, &l0);
  const float m_use = (mx == kNegInf) ? 0.0f : mx;
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  float wsum = 0.0f;
  for (int b0 = 0; warp + kWideWarps * b0 < n; b0 += kWideBatch) {
    if (b0 > 0) {
#pragma unroll
      for (int i = 0; i < kWideBatch; ++i) {
        const int s = warp + kWideWarps * (b0 + i);
        if (s < n) {
          va[i] = __ldcg(cols(s));
          vb[i] = __ldcg(cols(s) + 1);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kWideBatch; ++i) {
      const int s = warp + kWideWarps * (b0 + i);
      if (s >= n) break;
      const float w = piece_weight(p.part_lse, s, l0, m_use, prow);
      wsum += w;
      acc[0] += w * va[i].x; acc[1] += w * va[i].y; acc[2] += w * va[i].z; acc[3] += w * va[i].w;
      acc[4] += w * vb[i].x; acc[5] += w * vb[i].y; acc[6] += w * vb[i].z; acc[7] += w * vb[i].w;
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) part[warp][8 * lane + e] = acc[e];
  if (lane == 0) part_w[warp] = wsum;
  __syncthreads();
  if (warp != 0) return;
  float tot[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  float wtot = 0.0f;
#pragma unroll
  for (int q = 0; q < kWideWarps; ++q) {
    wtot += part_w[q];
#pragma unroll
    for (int e = 0; e < 8; ++e) tot[e] += part[q][8 * lane + e];
  }
  const float inv = wtot > 0.0f ? 1.0f / wtot : 0.0f;
  uint4 o;
  o.x = ptx::pack_bf16x2(tot[0] * inv, tot[1] * inv);
  o.y = ptx::pack_bf16x2(tot[2] * inv, tot[3] * inv);
  o.z = ptx::pack_bf16x2(tot[4] * inv, tot[5] * inv);
  o.w = ptx::pack_bf16x2(tot[6] * inv, tot[7] * inv);
  const size_t orow = static_cast<size_t>(sq.q_start + tok) * kQHeads + kGroup * g + row % kGroup;
  if (!row_ok(static_cast<long long>(orow), p.out_rows, p.status)) return;
  *reinterpret_cast<uint4*>(p.out + orow * kHeadDim + 8 * lane) = o;
  if (lane == 0 && p.lse != nullptr)
    p.lse[orow] = wtot > 0.0f ? (m_use + __log2f(wtot)) * kLn2 : kNegInf;
}

}  // namespace

size_t fwd_smem_bytes() { return kSmemAlloc; }

cudaError_t prepare_fwd_kernel() {
  const void* kernels[] = {
      reinterpret_cast<const void*>(gqa_attn_fwd_sm103_kernel<false, 0, 0>),
      reinterpret_cast<const void*>(gqa_attn_fwd_sm103_kernel<true, 0, 0>),
      reinterpret_cast<const void*>(gqa_attn_fwd_sm103_kernel<false, 1, 0>),
      reinterpret_cast<const void*>(gqa_attn_fwd_sm103_kernel<true, 1, 0>),
      reinterpret_cast<const void*>(gqa_attn_fwd_sm103_kernel<false, 2, 0>),
      reinterpret_cast<const void*>(gqa_attn_fwd_sm103_kernel<true, 2, 0>),
      reinterpret_cast<const void*>(gqa_attn_fwd_sm103_kernel<false, 0, 1>),
      reinterpret_cast<const void*>(gqa_attn_fwd_sm103_kernel<true, 0, 1>),
      reinterpret_cast<const void*>(gqa_attn_fwd_sm103_kernel<false, 1, 1>),
      reinterpret_cast<const void*>(gqa_attn_fwd_sm103_kernel<true, 1, 1>),
      reinterpret_cast<const void*>(gqa_attn_fwd_sm103_kernel<false, 2, 1>),
      reinterpret_cast<const void*>(gqa_attn_fwd_sm103_kernel<true, 2, 1>),
      reinterpret_cast<const void*>(gqa_attn_fwd_sm103_kernel<false, 0, 2>),
      reinterpret_cast<const void*>(gqa_attn_fwd_sm103_kernel<true, 0, 2>)};
  for (const void* f : kernels) {
    const cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(kSmemAlloc));
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

namespace {
// Launch configuration with programmatic dependent launch allowed (the kernels
// wait with griddepcontrol.wait before touching global memory) and, for CTA
// pairs, clusters of two.
cudaLaunchConfig_t launch_config(dim3 grid, dim3 block, size_t smem, bool pair,
                                 cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 1;
  if (pair) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  cfg.attrs = attr;
  return cfg;
}
}  // namespace

cudaError_t max_active_pairs(int* pairs) {
  // The smallest count over the pair kernels' block sizes: 4 softmax warps (dense),
  // 8 (quantised PV), 4 with the second TMA warp (paged).
  struct Shape {
    int fp8, kv;
    void (*kernel)(FwdParams);
  };
  const Shape shapes[3] = {{0, 0, gqa_attn_fwd_sm103_kernel<true, 0, 0>},
                           {2, 0, gqa_attn_fwd_sm103_kernel<true, 0, 2>},
                           {0, 1, gqa_attn_fwd_sm103_kernel<true, 1, 0>}};
  int best = 1 << 30;
  for (const Shape& sh : shapes) {
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = launch_config(dim3(2), dim3(fwd_threads(sh.fp8, sh.kv)), kSmemAlloc,
                                           true, nullptr, attr);
    cfg.attrs = attr + 1;  // occupancy of the cluster shape only
    cfg.numAttrs = 1;
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, sh.kernel, &cfg);
    if (e != cudaSuccess) return e;
    best = std::min(best, n);
  }
  *pairs = best;
  return cudaSuccess;
}

template <bool kPair>
cudaError_t launch_fwd_of(const cudaLaunchConfig_t& cfg, const FwdParams& p, int kv, int fp8) {
  if (fp8 == 2) return cudaLaunchKernelEx(&cfg, gqa_attn_fwd_sm103_kernel<kPair, 0, 2>, p);
  switch (kv * 2 + fp8) {
    case 0: return cudaLaunchKernelEx(&cfg, gqa_attn_fwd_sm103_kernel<kPair, 0, 0>, p);
    case 1: return cudaLaunchKernelEx(&cfg, gqa_attn_fwd_sm103_kernel<kPair, 0, 1>, p);
    case 2: return cudaLaunchKernelEx(&cfg, gqa_attn_fwd_sm103_kernel<kPair, 1, 0>, p);
    case 3: return cudaLaunchKernelEx(&cfg, gqa_attn_fwd_sm103_kernel<kPair, 1, 1>, p);
    case 4: return cudaLaunchKernelEx(&cfg, gqa_attn_fwd_sm103_kernel<kPair, 2, 0>, p);
    default: return cudaLaunchKernelEx(&cfg, gqa_attn_fwd_sm103_kernel<kPair, 2, 1>, p);
  }
}

cudaError_t launch_fwd(const FwdParams& p, int grid, bool pair, int kv, int fp8,
                       cudaStream_t stream) {
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg =
      launch_config(dim3(static_cast<unsigned>(grid)), dim3(fwd_threads(fp8, kv)), kSmemAlloc,
                    pair, stream, attr);
  return pair ? launch_fwd_of<true>(cfg, p, kv, fp8) : launch_fwd_of<false>(cfg, p, kv, fp8);
}

cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream) {
  if (p.tail_items < 1 || p.tail_splits == 1) return cudaSuccess;
  // Merged row rr of an item holds token 21 * (ctas_per_item * qt + rr / 126) + (rr % 126) / 6
  // = tok_per_item * qt + rr / 6 >= rr / 6, so only rows rr < 6 * (longest chunk) can be live:
  // a decode-sized call launches 6 to 24 rows per item, not 126 or 252.
  int max_q = 0;
  for (int i = 0; i < p.batch.n_seq; ++i) max_q = std::max(max_q, p.batch.seq[i].q_len);
  const int rows = std::min(p.ctas_per_item * kTokPerTile * kGroup, kGroup * max_q);
  if (rows < 1) return cudaSuccess;
  cudaLaunchAttribute attr[2];
  // Pieces per tail item: S, or for the balanced tail about workers / items + 1.
  const int pieces = p.tail_splits > 0 ? p.tail_splits : p.workers / p.tail_items + 1;
  if (pieces >= kWideMergePieces) {  // many pieces per item: a block per row
    const dim3 grid(static_cast<unsigned>(p.tail_items), static_cast<unsigned>(rows));
    const cudaLaunchConfig_t cfg = launch_config(grid, dim3(kWideWarps * 32), 0, false, stream, attr);
    return cudaLaunchKernelEx(&cfg, merge_wide_kernel, p);
  }
  const dim3 grid(static_cast<unsigned>(p.tail_items),
                  static_cast<unsigned>((rows + kMergeRowsPerBlock - 1) / kMergeRowsPerBlock));
  const cudaLaunchConfig_t cfg = launch_config(grid, dim3(256), 0, false, stream, attr);
  return cudaLaunchKernelEx(&cfg, merge_tail_kernel, p);
}

cudaError_t status_word_address(int** ptr) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(ptr), g_status_word);
}

}  // namespace gqa
