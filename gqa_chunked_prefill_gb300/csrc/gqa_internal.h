// Internal interface between the host library (gqa_prefill_host.cu) and the
// device kernels (attn_fwd_sm103.cu). Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gqa_schedule.h"

namespace gqa {

// Fixed problem geometry (the only shape the library accepts).
constexpr int kHeadDim = 256;
constexpr int kQHeads = 24;
constexpr int kKvHeads = 4;
constexpr int kGroup = kQHeads / kKvHeads;  // 6 query heads per KV head
// One MMA M tile of 128 rows holds 21 tokens x 6 heads = 126 rows (+2 idle rows).
constexpr int kTokPerTile = 21;
constexpr int kRowsPerTile = 128;
constexpr int kBlockN = 128;  // keys per KV tile

// Softmax warps of the attention kernel (fp8: 0 BF16, 1 FP8 QK^T, 2 FP8 QK^T and
// PV): 4, one thread per MMA row; with quantised PV 8, two threads per row on 64
// of a tile's 128 scores each. Then the TMA warp, two MMA-issuing warps (QK^T,
// PV) and, for paged K/V (kv == 1), a second TMA warp for the V ring.
constexpr int fwd_softmax_warps(int fp8) { return fp8 == 2 ? 8 : 4; }
constexpr bool fwd_split_producer(int kv) { return kv == 1; }
constexpr int fwd_threads(int fp8, int kv) {
  return (fwd_softmax_warps(fp8) + (fwd_split_producer(kv) ? 4 : 3)) * 32;
}

struct FwdParams {
  CUtensorMap tmap_q;  // Q [q_len][24][256], box (64 d, 6 heads, 21 tokens), 128B swizzle
  // K, V boxes of one stage (per CTA): K 128 keys x 2 chunks of 64 d (pairs: 64 x 4),
  // V 64 keys x 4 chunks (pairs: 128 x 2). Dense K/V [kv_len][4][256]: 4-D maps
  // (64 d, key, head, chunk); paged caches: 5-D maps (64 d, key % 8, chunk, key / 8,
  // head) over all num_pages * page_size rows (stage layouts: attn_fwd_sm103.cu).
  CUtensorMap tmap_k;
  CUtensorMap tmap_v;
  __nv_bfloat16* out;  // [q_len][24][256]
  float* lse;          // [q_len][24] natural log, or null
  float* part_o;       // [slots][128 rows][256] normalised partial O of split pieces
  float* part_lse;     // [slots][128 rows] base-2 partial LSE (slots: gqa_schedule.h)
  int* status;         // per-device status word
  long long out_rows;  // rows of 256 values in out / entries of lse (bounds-checked build)
  long long part_rows; // rows in part_o / part_lse (bounds-checked build)
  int head_items;      // Schedule (gqa_schedule.h): items processed whole first
  int tail_splits;     //   pieces per remaining item (0: balanced tail)
  int n_units;         //   units dealt to the CTAs (uniform tail)
  int n_tail;          //   tail items (balanced tail)
  float scale_log2;    // scale * log2(e)
  unsigned long long timeout_ns;
  int withhold_q;      // test only: the producer never loads the first Q tile
  int kv_read_once;    // no KV tile is read by two items (decode-sized chunks)
  // Paged K/V (kernels instantiated with kPaged only): key j of the sequence is
  // cache row block_table[j / page_size] * page_size + j % page_size (gqa_paged.h).
  CUtensorMap tmap_k_sub;    // 5-D, sub_rows keys x the stage's chunks: pieces of a box
  CUtensorMap tmap_v_sub;    //   that crosses a page
  CUtensorMap tmap_v16;      // 16 keys: V of the tile holding key kv_len-1 (paged: 5-D, all
                             //   the stage's chunks; dense batch: 4-D, one chunk)
  const int* block_table;    // sequence b's row at b * bt_stride: physical page of each
  int bt_stride;             //   logical page (ceil(kv_len_b / page_size) used entries)
  int page_size;             // keys per page, a multiple of 16
  int num_pages;             // pages in the cache
  int sub_rows;              // gcd(page_size, 64)
  int oob_row;               // a row past the cache (num_pages * page_size) or, for a dense
                             //   batch, past the packed K/V (total keys): TMA zero fill
  // FP8 QK^T (kernels instantiated with kFp8 only): tmap_q / tmap_k hold E4M3 codes
  // (Q box (128, 6 heads, 21 tokens); K 4-D (128, key, head, chunk) with 2 chunks).
  CUtensorMap tmap_ks;       // dense: key scales FP32 [4][k_scale_stride], box (128 keys, 1 head)
  const float* k_scale;      // paged: one scale per cache row, [4][k_scale_stride], read by
  int k_scale_stride;        //   1-D bulk copies (16-key pieces are 64 bytes)
  const float* q_scale;      // [total q rows][24] FP32 query scales
  // Quantised PV (kernels instantiated with kFp8 = 2): tmap_v holds V's E4M3 codes
  // transposed, [4 heads][256 channels][v_stride keys] bytes, 3-D (key, channel,
  // head), box (128 keys, 256 channels or a pair CTA's 128, 1 head), 128B swizzle.
  const float* v_scale;      // [4][256] FP32 per-channel scales of V
  TailPrefix tail;           // balanced tail: tile prefix sums of the tail items
  Batch batch;               // the call's sequences (gqa_schedule.h); kept last: it is large
};

struct MergeParams {
  const float* part_o;    // as FwdParams::part_o
  const float* part_lse;  // as FwdParams::part_lse
  __nv_bfloat16* out;
  float* lse;             // may be null
  int* status;            // per-device status word
  long long out_rows;     // as FwdParams (bounds-checked build)
  long long part_rows;
  int head_items;
  int tail_items;         // one merge block column per tail item
  int tail_splits;        // S > 1 (uniform), or 0 (balanced: pieces from `tail`)
  int workers;            // balanced: the attention grid's CTAs (or pairs)
  int ctas_per_item;      // 1, or 2 for the CTA-pair kernel (42-token items)
  TailPrefix tail;        // as FwdParams::tail
  Batch batch;            // as FwdParams::batch
};

size_t fwd_smem_bytes();
// grid = CTAs; with pair = true the CTAs form clusters of two (grid even).
// kv: 0 dense K/V of one sequence, 1 paged K/V, 2 dense K/V of a batch;
// fp8: 0 BF16, 1 E4M3 QK^T, 2 E4M3 QK^T and PV (dense K/V of one sequence).
cudaError_t launch_fwd(const FwdParams& p, int grid, bool pair, int kv, int fp8,
                       cudaStream_t stream);
// Scale column of each key row for head-major key scales: sequence b of a packed
// batch (rows row_begin[b] .. row_begin[b+1]-1) starts at column col_begin[b].
struct ScaleColumns {
  int n_seq;  // 1: column = row
  int row_begin[kMaxSeqs + 1];
  int col_begin[kMaxSeqs];
};
// E4M3 codes and scales of rows x heads vectors of 256 BF16 values (quantize_fp8.cu);
// num_sms sizes the persistent grid.
cudaError_t launch_quantize_fp8(const void* x, void* codes, float* scale, int rows, int heads,
                                int scale_stride, bool head_major, const ScaleColumns& cols,
                                int num_sms, cudaStream_t stream);
// E4M3 codes of V transposed to [4][256][v_stride] and per-(head, channel) scales
// [4][256] (quantize_fp8.cu).
cudaError_t launch_quantize_v_fp8(const void* v, void* codes, float* scale, int kv_len,
                                  int v_stride, cudaStream_t stream);
cudaError_t max_active_pairs(int* pairs);       // co-resident CTA pairs on this device

cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream);
cudaError_t prepare_fwd_kernel();                // per-device one-time attributes
cudaError_t status_word_address(int** ptr);      // device address of the status word

}  // namespace gqa
