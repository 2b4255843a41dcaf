// Per-vector FP8 (E4M3) quantisation of Q and K for the quantised-QK^T path.
//
// Method (gfx936 DCU上实现INT8 QK MMAC：分页访存、Fragment映射与GQA适配, §1 and §4):
// each query vector (token, query head) and each key vector (token, KV head)
// of head_dim values gets one symmetric dynamic scale, s = max|x| / qmax, and
// codes x / s; the scores are restored as code_q . code_k * s_q * s_k * scale
// before the softmax. The report quantises to INT8 (qmax 127) for gfx936's
// INT8 MMAC. On GB300 the native low-precision tensor path is FP8, so the codes
// are E4M3 (qmax 448, round to nearest even, saturating); Q is quantised once,
// before attention, like the report's producer-side Q quantisation (§4).
//
// Key scales are stored head-major, [4][stride]; in a batch packed end to end,
// sequence b's scales start at column col_begin[b] (a multiple of 4, so that
// the attention kernel's TMA copies of them start on 16 bytes) instead of at
// its first key row.
//
// Every rounding decision is taken in FP32 exactly as written: s = amax / 448
// and x / s are IEEE round-to-nearest divisions (no reciprocal), then one
// RNE conversion to E4M3. A vector of zeros gets s = 0 and codes 0.
//
// One warp per vector of 256 BF16 values (16 bytes per lane): HBM-bound, one
// read of the BF16 input and one write of the codes and the scale.

#include "gqa_internal.h"
#include "sm100_ptx.cuh"

namespace gqa {
namespace {

constexpr float kE4m3Max = 448.0f;
constexpr int kVecPerBlock = 8;  // 8 warps

__global__ void __launch_bounds__(256)
    quantize_fp8_kernel(const __nv_bfloat16* __restrict__ x, uint8_t* __restrict__ codes,
                        float* __restrict__ scale, int n_vec, int heads, int scale_stride,
                        int head_major, const __grid_constant__ ScaleColumns cols) {
  const int vec = blockIdx.x * kVecPerBlock + static_cast<int>(threadIdx.x >> 5);
  if (vec >= n_vec) return;  // whole warps leave together
  const int lane = threadIdx.x & 31;
  const uint4 raw = reinterpret_cast<const uint4*>(x + static_cast<size_t>(vec) * kHeadDim)[lane];
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  float v[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // BF16 -> FP32 is exact: the BF16 bits are the top half
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = __fdiv_rn(amax, kE4m3Max);
  uint32_t packed[2] = {0u, 0u};
  if (s > 0.0f) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t pair = ptx::cvt_e4m3x2(__fdiv_rn(v[2 * i], s), __fdiv_rn(v[2 * i + 1], s));
      packed[i >> 1] |= pair << (16 * (i & 1));
    }
  }
  reinterpret_cast<uint2*>(codes + static_cast<size_t>(vec) * kHeadDim)[lane] =
      make_uint2(packed[0], packed[1]);
  if (lane == 0) {
    const int row = vec / heads, h = vec - (vec / heads) * heads;
    int col = row;  // head-major: the scale column of this row (sequences start on 4)
    if (head_major && cols.n_seq > 1) {
      int lo = 0, hi = cols.n_seq - 1;  // the last sequence starting at or before `row`
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cols.row_begin[mid] <= row) lo = mid;
        else hi = mid - 1;
      }
      col = cols.col_begin[lo] + row - cols.row_begin[lo];
    }
    scale[head_major ? static_cast<size_t>(h) * scale_stride + col
                     : static_cast<size_t>(row) * heads + h] = s;
  }
}

}  // namespace

cudaError_t launch_quantize_fp8(const void* x, void* codes, float* scale, int rows, int heads,
                                int scale_stride, bool head_major, const ScaleColumns& cols,
                                cudaStream_t stream) {
  const int n_vec = rows * heads;
  if (n_vec == 0) return cudaSuccess;
  const int blocks = (n_vec + kVecPerBlock - 1) / kVecPerBlock;
  quantize_fp8_kernel<<<blocks, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(x),
                                                   static_cast<uint8_t*>(codes), scale, n_vec,
                                                   heads, scale_stride, head_major ? 1 : 0, cols);
  return cudaGetLastError();
}

}  // namespace gqa
