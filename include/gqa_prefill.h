/*
 * gqa_prefill.h — C ABI of the GB300 (sm_103a) chunked-prefill causal GQA
 * attention library (libgqa_prefill.so).
 *
 * The operation (DCU使用技术报告（中篇）：gfx936 DCU上的Qwen3.5-27B Triton-ROCm
 * Attention与GEMV深度优化实战, §2 "专用 Prefill Attention"): one sequence, BF16,
 * 24 query heads / 4 KV heads / head_dim 256 (GQA ratio 6, same report §1);
 * QK^T, causal mask, online softmax and PV with FP32 accumulation. Query head h
 * reads KV head h/6 (gfx936 DCU上实现INT8 QK MMAC：分页访存、Fragment映射与GQA适配,
 * §5.2). The q_len new tokens of the chunk sit at the END of the kv_len-long
 * K/V prefix (the prefix already holds the chunk's own keys), so query token t
 * has absolute position kv_len - q_len + t and sees keys 0 .. kv_len - q_len + t
 * (DCU report, §3: later chunks of a request see a longer kv_len).
 *
 * Shapes outside that contract are refused, never silently mapped (DCU report
 * §2: unsupported shapes fall back; INT8 QK MMAC page §7: wrong layouts are
 * rejected rather than run with a wrong mapping). This library has no fallback:
 * a refused call returns an error code and launches nothing.
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE memory on the current CUDA device, owned
 *    by the caller; the library keeps no reference after the call returns.
 *  - Tensors are dense, row-major, no padding:
 *        q, out : [q_len,  n_q_heads,  head_dim]  BF16
 *        k, v   : [kv_len, n_kv_heads, head_dim]  BF16
 *        lse    : [q_len,  n_q_heads]             FP32, natural log
 *    Every pointer must be 16-byte aligned (the kernels move tiles with TMA).
 *  - `stream` is a cudaStream_t (CUstream) handle; NULL means the legacy
 *    default stream. Calls are asynchronous on that stream: they return as
 *    soon as the work is queued. Any temporary device memory is allocated and
 *    freed in stream order on `stream`.
 *  - Errors found on the host are returned before anything is launched. A
 *    device-side wait that exceeds its time limit makes the kernel give up,
 *    record GQA_ERR_DEVICE_TIMEOUT in a per-device status word and return;
 *    read it with gqa_prefill_poll().
 */
#ifndef GQA_PREFILL_H_
#define GQA_PREFILL_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GQA_PREFILL_ABI_VERSION 12

typedef enum gqa_status {
  GQA_OK = 0,
  GQA_ERR_NULL = 1,           /* a required pointer is NULL                           */
  GQA_ERR_SHAPE = 2,          /* q_len < 0, kv_len < q_len, kv_len == 0 with q_len > 0,
                                 or scale not finite and > 0                            */
  GQA_ERR_UNSUPPORTED = 3,    /* head counts / head_dim other than 24 / 4 / 256, or no
                                 sm_103a-class device                                  */
  GQA_ERR_ALIGN = 4,          /* a pointer is not 16-byte aligned                      */
  GQA_ERR_CUDA = 5,           /* a CUDA runtime/driver call failed                     */
  GQA_ERR_DEVICE_TIMEOUT = 6, /* a device-side wait ran out of time (see _poll)        */
  GQA_ERR_SCRATCH = 7,        /* gqa_prefill_attn_noalloc: the call's split partials do
                                 not fit the library's static scratch array            */
  GQA_ERR_PAGE_TABLE = 8,     /* device-side (see _poll): a paged call met a block-table
                                 entry outside [0, num_pages); that page read as zeros */
  GQA_ERR_BOUNDS = 9          /* device-side, bounds-checked build only (libgqa_prefill_checked.so,
                                 see _poll): an output, LSE or split-partial index fell outside
                                 its buffer; the access was skipped                     */
} gqa_status;

/*
 * out[t, h, :] = softmax_j( scale * q[t,h,:] . k[j, h/6, :] ) v[j, h/6, :],
 *                j = 0 .. kv_len - q_len + t
 * lse[t, h]    = ln sum_j exp( scale * q[t,h,:] . k[j, h/6, :] )   (same j range)
 *
 * q_len == 0 returns GQA_OK without launching. `lse` may be NULL.
 * `scale` is used as given (1/sqrt(head_dim) = 1/16 for this model); it must
 * be finite and > 0.
 */
gqa_status gqa_prefill_attn(const void* q, const void* k, const void* v, void* out, float* lse,
                            int q_len, int kv_len, int n_q_heads, int n_kv_heads, int head_dim,
                            float scale, void* stream);

/* gqa_prefill_opts.force_splits (and the make_plan calls' force_splits): cut the
   tail in the balanced form (see gqa_prefill_plan). */
#define GQA_FORCE_BALANCED_TAIL (-1)

/* Options for gqa_prefill_attn_ex (zero-initialise; zero fields mean "default"). */
typedef struct gqa_prefill_opts {
  int force_splits;           /* 0: planner decides; S > 0: every full round of the
                                 grid takes whole items and each remaining item is
                                 split into S KV pieces (capped at the shortest
                                 item's tile count; 1 = no split, no merge pass);
                                 GQA_FORCE_BALANCED_TAIL: the balanced tail (the
                                 planner's best number of whole rounds for it), or
                                 the planner's choice where no tail fits it      */
  int force_grid;             /* > 0: use at most this many CTAs (tests use it to cut
                                 items into many pieces); 0: one CTA per SM       */
  uint32_t wait_timeout_us;   /* bound on any single device-side wait; 0 = 2 s      */
  void* fwd_event_begin;      /* optional cudaEvent_t recorded on `stream` right
                                 before the attention kernel launch                */
  void* fwd_event_end;        /* optional cudaEvent_t recorded right after it (before
                                 the split merge, if any): times the main kernel   */
  int test_withhold_q;        /* TEST ONLY. 1: the TMA producer withholds each CTA's
                                 first Q tile, so every consumer wait runs out after
                                 wait_timeout_us; the kernel records
                                 GQA_ERR_DEVICE_TIMEOUT, drains its copies, frees
                                 tensor memory and returns (outputs undefined).
                                 Exercises the time-out path without faulting.     */
  int force_variant;          /* 0: planner decides; 1: one CTA per 21-token item;
                                 2: a CTA pair per 42-token item (cta_group::2 MMAs) */
  int reserved[1];
} gqa_prefill_opts;

/*
 * What the planner chose (the route check: which kernel ran and how).
 * A work item is one 21-token query tile of one KV group (21 x 6 = 126 MMA
 * rows); it visits KV tiles of 128 keys up to the causal diagonal. Items are
 * ordered longest first and dealt to the persistent CTAs in a snake, whole
 * items in the first head_rounds full rounds. The remaining (tail) items are
 * cut in one of two ways: uniform, each split into tail_splits pieces of equal
 * KV length; or balanced (tail_splits == 0), their tiles laid end to end and
 * every CTA (pair) taking an equal share, cut at item boundaries. A second
 * kernel merges the pieces of every split item.
 */
typedef struct gqa_prefill_plan {
  int num_sms;                /* SMs of the device                                    */
  int q_tiles;                /* ceil(q_len / tokens per item), summed over sequences */
  int n_items;                /* q_tiles * n_kv_heads                                 */
  int head_rounds;            /* full rounds of whole items                           */
  int tail_items;             /* items after those rounds                             */
  int tail_splits;            /* KV pieces per tail item (1 = whole, no merge pass);
                                 0 = balanced tail                                    */
  int n_units;                /* pieces computed: head items + tail_items * tail_splits
                                 (balanced: head items + the tail's pieces)          */
  int grid;                   /* CTAs launched for the attention kernel               */
  int kernels_per_call;       /* launches per call: 1, or 2 with the merge kernel     */
  int variant;                /* 1 = one CTA per item (M = 128 MMAs, 21 tokens);
                                 2 = a CTA pair per item (cta_group::2, M = 256, 42
                                 tokens: each CTA streams half of every K/V tile)  */
  int64_t total_tiles;        /* KV tiles summed over all items                       */
  int64_t workspace_bytes;    /* temporary device memory of the split items (or 0):
                                 FP32 partials, 128 rows x 257 floats per CTA of an
                                 item (cpi = 1, or 2 for the CTA pair) per slot, in
                                 tail_items * tail_splits slots (uniform tail) or 2
                                 slots per worker (balanced tail: workers = grid /
                                 cpi), i.e. slots * cpi * 128 * 1028 bytes         */
  int64_t est_makespan_tiles; /* planner's cost of the busiest CTA, in KV tiles       */
} gqa_prefill_plan;

/* gqa_prefill_attn with options; `opts` and `plan_out` may each be NULL. */
gqa_status gqa_prefill_attn_ex(const void* q, const void* k, const void* v, void* out, float* lse,
                               int q_len, int kv_len, int n_q_heads, int n_kv_heads, int head_dim,
                               float scale, void* stream, const gqa_prefill_opts* opts,
                               gqa_prefill_plan* plan_out);

/*
 * Host-only planning (no CUDA call): fills *plan for a device with `num_sms`
 * SMs of which `max_pairs` CTA pairs of the pair kernel can be resident at
 * once, exactly as gqa_prefill_attn_ex would with the same force_* options
 * (0 = planner decides). max_pairs < 0 assumes num_sms / 2; larger values are
 * capped there; 0 plans without the pair kernel. gqa_prefill_device_info gives
 * both numbers for the current device, so a plan made from them is the plan
 * the attention call runs there. Validates shapes like the attention call
 * (pointers are not involved).
 */
gqa_status gqa_prefill_make_plan(int q_len, int kv_len, int n_q_heads, int n_kv_heads, int head_dim,
                                 int num_sms, int max_pairs, int force_splits, int force_grid,
                                 int force_variant, gqa_prefill_plan* plan);

/*
 * The planner's inputs on the CURRENT device, as the attention calls use them:
 * its SM count and the number of CTA pairs of the pair kernel that can be
 * resident at once (cudaOccupancyMaxActiveClusters, at most num_sms / 2; 0 if
 * the pair kernel cannot run). Does the library's one-time per-device set-up on
 * first use (make that first call outside any stream capture). Either pointer
 * may be NULL. GQA_ERR_UNSUPPORTED on a device that is not sm_103.
 */
gqa_status gqa_prefill_device_info(int* num_sms, int* max_pairs);

/*
 * Synchronises `stream`, then reads and clears the current device's status
 * word (0, GQA_ERR_DEVICE_TIMEOUT or GQA_ERR_PAGE_TABLE) into *device_status. Returns GQA_ERR_CUDA
 * if the synchronisation itself fails. The status word is shared by all
 * streams of the device: it reports any kernel of this library that gave up
 * since the previous poll.
 */
gqa_status gqa_prefill_poll(void* stream, int* device_status);

/*
 * gqa_prefill_attn_noalloc — same operation, arguments and results as
 * gqa_prefill_attn, but it allocates no device memory at all. (The subject
 * pages have no counterpart to this entry point; it exists for callers of this
 * library, not for the method.)
 *
 * Who needs it: callers that cannot allocate device memory in the middle of a
 * call — serving engines that reserve the whole device-memory budget at
 * start-up and forbid later allocations, code that must never risk the
 * implicit device-wide synchronisation a cudaFree can cause, and hosts whose
 * device allocator is owned by another framework. gqa_prefill_attn takes its
 * split-KV partials from a stream-ordered pool; this variant takes them from a
 * fixed scratch array compiled into the library instead.
 *
 * The scratch array is GQA_NOALLOC_SCRATCH_BYTES (64 MiB) of device memory,
 * held on every GPU that loads the library until the process exits. The call
 * plans exactly like gqa_prefill_attn; when that plan's workspace_bytes (see
 * gqa_prefill_plan: for a uniform tail tail_items * tail_splits * cpi * 128 *
 * 1028 bytes, for a balanced tail 2 * workers * cpi * 128 * 1028 bytes — at
 * most about 40 MB on 152 SMs; cpi = 2 for CTA-pair plans) exceed the array,
 * it returns GQA_ERR_SCRATCH and launches nothing.
 *
 * It calls no cudaMalloc, cudaFree or other allocating routine. Its first call
 * on each device does a one-time set-up with that device current (device
 * check, kernel attributes, and cudaGetSymbolAddress of the scratch array and
 * the status word); make that first call before any stream capture. Every
 * call shares the one array and it keeps the last call's contents (nothing in
 * it needs to start at zero: every partial row is written before it is read):
 * calls whose work overlaps on the GPU — on
 * different streams, or in different threads without ordering between them —
 * race on it and give undefined results. Serialise such calls.
 */
#define GQA_NOALLOC_SCRATCH_BYTES (64ull << 20)
gqa_status gqa_prefill_attn_noalloc(const void* q, const void* k, const void* v, void* out,
                                    float* lse, int q_len, int kv_len, int n_q_heads,
                                    int n_kv_heads, int head_dim, float scale, void* stream);

/*
 * gqa_prefill_attn_paged — the same operation with K and V read from a paged
 * cache instead of dense [kv_len, ...] arrays (gfx936 DCU上实现INT8 QK MMAC：
 * 分页访存、Fragment映射与GQA适配, §3: a logical key token is found through the
 * block table, which gives its physical block, and its slot inside that block;
 * DCU使用技术报告（中篇）, §8: the serving engine's BF16 attention page holds 784
 * tokens).
 *
 *   k_cache, v_cache : BF16 [num_pages, page_size, n_kv_heads, head_dim], dense
 *   block_table      : int32 [ceil(kv_len / page_size)], DEVICE memory: logical
 *                      key j (0 <= j < kv_len) of the sequence is row
 *                      j % page_size of page block_table[j / page_size]
 *
 * q, out, lse, scale and the causal alignment are those of gqa_prefill_attn:
 * the chunk's q_len tokens are the last q_len of the kv_len keys, whose K/V are
 * already in the cache. Pages may be listed in any order and shared between
 * sequences. Rows of the last page past kv_len may hold anything, NaN
 * included: they never reach the output.
 *
 * Requirements (else an error, nothing launched): page_size a positive
 * multiple of 16 (GQA_ERR_UNSUPPORTED); num_pages >= 1 and
 * num_pages * page_size < 2^30 (TMA row coordinates are 32-bit; 2^30 rows
 * would be 2 TiB per cache; GQA_ERR_SHAPE); block_table non-NULL and 4-byte aligned, the other pointers
 * 16-byte aligned. The block table is read on the device: an entry outside
 * [0, num_pages) is not followed — the page's keys and values are read as
 * zeros and GQA_ERR_PAGE_TABLE is recorded in the status word (_poll).
 */
gqa_status gqa_prefill_attn_paged(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_table, int num_pages, int page_size,
                                  void* out, float* lse, int q_len, int kv_len, int n_q_heads,
                                  int n_kv_heads, int head_dim, float scale, void* stream);

/* gqa_prefill_attn_paged with options and the plan (as gqa_prefill_attn_ex).
 * Paged calls (this one and the paged batch calls) plan like the dense calls
 * except that, when force_variant is 0, they prefer the CTA-pair kernel: its
 * paged tiles run within a few percent of its dense ones, the one-CTA kernel's
 * do not. So a paged call's plan equals gqa_prefill_make_plan's for the same
 * shape only where both choose the same variant (force_variant set, or the
 * pair winning on dense K/V too). */
gqa_status gqa_prefill_attn_paged_ex(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_table, int num_pages, int page_size,
                                     void* out, float* lse, int q_len, int kv_len,
                                     int n_q_heads, int n_kv_heads, int head_dim, float scale,
                                     void* stream, const gqa_prefill_opts* opts,
                                     gqa_prefill_plan* plan_out);

/*
 * Batched (varlen) calls: up to GQA_MAX_SEQS sequences of a serving batch in
 * one launch. Each sequence is a chunk exactly as in gqa_prefill_attn: its
 * q_len new tokens are the last q_len of its kv_len keys (the pages restrict
 * their kernel to one sequence, DCU使用技术报告（中篇）, §2; batching the chunks
 * of several requests is the step beside it in a server). Work items of all
 * sequences share the persistent grid; the plan is made on the host from the
 * real lengths, so the length arrays are HOST memory (a serving scheduler
 * knows them there) and are read during the call only.
 *
 * gqa_prefill_attn_varlen: packed tensors
 *   q, out   : [total_q,  24, 256] BF16; lse [total_q, 24] FP32 (may be NULL)
 *   k, v     : [total_kv,  4, 256] BF16
 *   cu_seqlens_q, cu_seqlens_k : HOST int32 [batch + 1], starting at 0 and
 *     non-decreasing: sequence b owns query rows cu_seqlens_q[b] ..
 *     cu_seqlens_q[b+1]-1 and key rows cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1,
 *     with q_len_b <= kv_len_b. Empty sequences are allowed.
 * gqa_prefill_attn_paged_varlen: q / out / lse packed as above; K/V caches as
 *   gqa_prefill_attn_paged; block_table DEVICE int32 [batch][bt_stride]
 *   (bt_stride >= every sequence's ceil(kv_len_b / page_size)); kv_lens HOST
 *   int32 [batch].
 * batch > GQA_MAX_SEQS returns GQA_ERR_UNSUPPORTED (split the batch).
 */
#define GQA_MAX_SEQS 128
gqa_status gqa_prefill_attn_varlen(const void* q, const void* k, const void* v, void* out,
                                   float* lse, const int32_t* cu_seqlens_q,
                                   const int32_t* cu_seqlens_k, int batch, int n_q_heads,
                                   int n_kv_heads, int head_dim, float scale, void* stream);
gqa_status gqa_prefill_attn_varlen_ex(const void* q, const void* k, const void* v, void* out,
                                      float* lse, const int32_t* cu_seqlens_q,
                                      const int32_t* cu_seqlens_k, int batch, int n_q_heads,
                                      int n_kv_heads, int head_dim, float scale, void* stream,
                                      const gqa_prefill_opts* opts, gqa_prefill_plan* plan_out);
gqa_status gqa_prefill_attn_paged_varlen(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_table, int bt_stride, int num_pages,
                                         int page_size, void* out, float* lse,
                                         const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                                         int batch, int n_q_heads, int n_kv_heads, int head_dim,
                                         float scale, void* stream);
gqa_status gqa_prefill_attn_paged_varlen_ex(const void* q, const void* k_cache,
                                            const void* v_cache, const int32_t* block_table,
                                            int bt_stride, int num_pages, int page_size,
                                            void* out, float* lse,
                                            const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                                            int batch, int n_q_heads, int n_kv_heads,
                                            int head_dim, float scale, void* stream,
                                            const gqa_prefill_opts* opts,
                                            gqa_prefill_plan* plan_out);
/* Host-only planning of a dense batched call (as gqa_prefill_make_plan). */
gqa_status gqa_prefill_make_plan_varlen(const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                        int batch, int n_q_heads, int n_kv_heads, int head_dim,
                                        int num_sms, int max_pairs, int force_splits,
                                        int force_grid, int force_variant, gqa_prefill_plan* plan);
/* Host-only planning of a paged call (gqa_prefill_attn_paged[_ex], one sequence:
 * batch 1, cu_seqlens_q {0, q_len}, kv_lens {kv_len}) or paged batch
 * (gqa_prefill_attn_paged_varlen[_ex]); kv_lens HOST int32 [batch]. Paged calls
 * prefer the CTA-pair kernel (see gqa_prefill_attn_paged_ex), so this can differ
 * from gqa_prefill_make_plan_varlen for the same lengths. Same arguments,
 * validation and errors as gqa_prefill_make_plan_varlen otherwise. */
gqa_status gqa_prefill_make_plan_paged_varlen(const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                                              int batch, int n_q_heads, int n_kv_heads,
                                              int head_dim, int num_sms, int max_pairs,
                                              int force_splits, int force_grid, int force_variant,
                                              gqa_prefill_plan* plan);

/*
 * Quantised QK^T (gfx936 DCU上实现INT8 QK MMAC：分页访存、Fragment映射与GQA适配, §1
 * "INT8 QK的量化和Scale恢复" and §4 "Query量化只做一次"). The report quantises each
 * query vector (token, query head) and each key vector (token, KV head) with
 * one symmetric dynamic scale, multiplies the integer codes, and restores
 * score = (code_q . code_k) * s_q * s_k * softmax_scale for every score BEFORE
 * the softmax. Its codes are INT8 for gfx936's INT8 MMAC; on GB300 the native
 * low-precision tensor path is FP8, so here the codes are E4M3:
 *
 *   s    = max_c |x[c]| / 448                  (FP32, IEEE round-to-nearest division)
 *   code = E4M3(x[c] / s)                      (FP32 division, then round to nearest
 *                                               even, saturating at +-448)
 *   a vector of zeros gets s = 0 and codes 0.
 *
 * PV stays BF16 (V is not quantised), as does the output.
 *
 * gqa_quantize_q_fp8: q BF16 [q_len][24][256] -> q_fp8 E4M3 [q_len][24][256]
 *   (one byte per value), q_scale FP32 [q_len][24]. Run once per chunk, before
 *   attention (the report's producer-side quantisation).
 * gqa_quantize_k_fp8: k BF16 [kv_len][4][256] -> k_fp8 E4M3 [kv_len][4][256],
 *   k_scale FP32 [4][k_scale_stride] (head-major: key j of KV head g at
 *   g * k_scale_stride + j), k_scale_stride >= kv_len and a multiple of 4 (so
 *   every head's row starts on 16 bytes). Run when keys enter the cache.
 * Both are asynchronous on `stream`; pointers 16-byte aligned (q_scale 4-byte).
 *
 * gqa_prefill_attn_fp8qk[_ex]: the attention of gqa_prefill_attn with Q and K
 * given as those codes and scales; v, out, lse, scale, causal alignment, plan
 * and options as gqa_prefill_attn[_ex]. The result is the attention of the
 * DEQUANTISED query and keys (code * s) computed like the BF16 path.
 */
gqa_status gqa_quantize_q_fp8(const void* q, void* q_fp8, float* q_scale, int q_len,
                              int n_q_heads, int head_dim, void* stream);
gqa_status gqa_quantize_k_fp8(const void* k, void* k_fp8, float* k_scale, int kv_len,
                              int n_kv_heads, int head_dim, int k_scale_stride, void* stream);
gqa_status gqa_prefill_attn_fp8qk(const void* q_fp8, const float* q_scale, const void* k_fp8,
                                  const float* k_scale, int k_scale_stride, const void* v,
                                  void* out, float* lse, int q_len, int kv_len, int n_q_heads,
                                  int n_kv_heads, int head_dim, float scale, void* stream);
gqa_status gqa_prefill_attn_fp8qk_ex(const void* q_fp8, const float* q_scale, const void* k_fp8,
                                     const float* k_scale, int k_scale_stride, const void* v,
                                     void* out, float* lse, int q_len, int kv_len, int n_q_heads,
                                     int n_kv_heads, int head_dim, float scale, void* stream,
                                     const gqa_prefill_opts* opts, gqa_prefill_plan* plan_out);

/*
 * Quantised QK^T for batched calls, dense or paged (the report's production
 * path reads its quantised K from a paged cache, gfx936 DCU上实现INT8 QK MMAC, §3).
 * q_fp8 / q_scale packed [total_q][24][256] / [total_q][24]; V and out as the
 * BF16 batched calls.
 *  - dense: k_fp8 packed [total_kv][4][256]; k_scale [4][k_scale_stride] where
 *    sequence b's scales start at column sum_{i<b} roundup4(kv_len_i) (every
 *    sequence starts on 16 bytes, as the kernel's TMA copies of them must);
 *    k_scale_stride >= sum_b roundup4(kv_len_b), a multiple of 4.
 *    gqa_quantize_k_fp8_varlen writes exactly this layout.
 *  - paged: k_cache_fp8 [num_pages][page_size][4][256] E4M3 codes, k_scale
 *    [4][k_scale_stride] holding the scale of every CACHE ROW (row = page *
 *    page_size + slot), k_scale_stride >= num_pages * page_size, a multiple of
 *    4 (gqa_quantize_k_fp8 over the cache viewed as [num_pages * page_size][4][256]
 *    writes exactly this); v_cache BF16 as gqa_prefill_attn_paged.
 */
gqa_status gqa_quantize_k_fp8_varlen(const void* k, void* k_fp8, float* k_scale,
                                     const int32_t* cu_seqlens_k, int batch, int n_kv_heads,
                                     int head_dim, int k_scale_stride, void* stream);
gqa_status gqa_prefill_attn_fp8qk_varlen_ex(const void* q_fp8, const float* q_scale,
                                            const void* k_fp8, const float* k_scale,
                                            int k_scale_stride, const void* v, void* out,
                                            float* lse, const int32_t* cu_seqlens_q,
                                            const int32_t* cu_seqlens_k, int batch, int n_q_heads,
                                            int n_kv_heads, int head_dim, float scale,
                                            void* stream, const gqa_prefill_opts* opts,
                                            gqa_prefill_plan* plan_out);
gqa_status gqa_prefill_attn_paged_fp8qk_varlen_ex(
    const void* q_fp8, const float* q_scale, const void* k_cache_fp8, const float* k_scale,
    int k_scale_stride, const void* v_cache, const int32_t* block_table, int bt_stride,
    int num_pages, int page_size, void* out, float* lse, const int32_t* cu_seqlens_q,
    const int32_t* kv_lens, int batch, int n_q_heads, int n_kv_heads, int head_dim, float scale,
    void* stream, const gqa_prefill_opts* opts, gqa_prefill_plan* plan_out);

/*
 * Quantised PV (the INT8 QK MMAC page, §6: the final submission multiplied P by V
 * in 8 bits as well, without saying how V or P are scaled). Reading for GB300's
 * FP8 tensor path:
 *   - V gets one symmetric scale per (KV head, channel) over the call's kv_len
 *     keys: s_v[g][c] = max_j |v[j][g][c]| / 448, codes E4M3(v / s_v) (the
 *     rounding rules of gqa_quantize_q_fp8, along the key axis); the scale
 *     multiplies column c of P.V after the product;
 *   - P is rounded to E4M3 as the MMA operand (stored as 2^6 * p, p at most 4
 *     times the running maximum, so it never saturates), while the softmax
 *     normaliser and the LSE keep the FP32 probabilities.
 * The result approximates the attention of the DEQUANTISED query, keys and
 * values; rounding P moves an output element by at most
 * sum_j (2^-4 p_j + 2^-16) |v_j| / sum_j p_j (p_j = exp(s_j - max s)).
 *
 * gqa_quantize_v_fp8: v BF16 [kv_len][4][256] -> v_fp8t E4M3 [4][256][v_stride]
 *   (channel rows of key codes, TRANSPOSED so that a 128-key tile is a K-major
 *   MMA operand; v_stride >= kv_len, a multiple of 16; entries past kv_len are
 *   not written), v_scale FP32 [4][256]. Asynchronous on `stream` (a memset and
 *   three small kernels). All of one call's keys share the channel scales.
 * gqa_prefill_attn_fp8qkpv[_ex]: gqa_prefill_attn_fp8qk with V given as those
 *   codes and scales. One sequence, dense K/V (GQA_ERR_UNSUPPORTED otherwise);
 *   out, lse, options and plan as gqa_prefill_attn_fp8qk[_ex].
 */
gqa_status gqa_quantize_v_fp8(const void* v, void* v_fp8t, float* v_scale, int kv_len,
                              int n_kv_heads, int head_dim, int v_stride, void* stream);
gqa_status gqa_prefill_attn_fp8qkpv(const void* q_fp8, const float* q_scale, const void* k_fp8,
                                    const float* k_scale, int k_scale_stride, const void* v_fp8t,
                                    const float* v_scale, int v_stride, void* out, float* lse,
                                    int q_len, int kv_len, int n_q_heads, int n_kv_heads,
                                    int head_dim, float scale, void* stream);
gqa_status gqa_prefill_attn_fp8qkpv_ex(const void* q_fp8, const float* q_scale, const void* k_fp8,
                                       const float* k_scale, int k_scale_stride,
                                       const void* v_fp8t, const float* v_scale, int v_stride,
                                       void* out, float* lse, int q_len, int kv_len,
                                       int n_q_heads, int n_kv_heads, int head_dim, float scale,
                                       void* stream, const gqa_prefill_opts* opts,
                                       gqa_prefill_plan* plan_out);

/* Static description of a status code (never NULL). */
const char* gqa_status_string(gqa_status status);

/* GQA_PREFILL_ABI_VERSION of the loaded library. */
int gqa_prefill_abi_version(void);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* GQA_PREFILL_H_ */
