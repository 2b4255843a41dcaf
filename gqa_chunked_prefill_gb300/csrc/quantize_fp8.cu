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
// is an IEEE round-to-nearest division and x / s is the round-to-nearest
// quotient (from the reciprocal of s and Markstein's correction, equal to the
// IEEE division for every BF16 input: fp8_quotient.cuh), then one RNE
// conversion to E4M3. A vector of zeros gets s = 0 and codes 0.
//
// A persistent grid (8 blocks of 8 warps per SM); each warp takes two
// vectors of 256 BF16 values at a time (16 bytes per lane each) and issues the
// loads of its next two before it works on the current ones: one read of the
// BF16 input and one write of the codes and the scale. The IEEE division per
// value made the first version issue-bound (three quarters of the issue slots
// busy at under half the HBM rate); the correction takes three packed FP32
// instructions per two values.

#include <algorithm>

#include "fp8_quotient.cuh"
#include "gqa_internal.h"
#include "sm100_ptx.cuh"

namespace gqa {
namespace {

constexpr float kE4m3Max = 448.0f;
constexpr int kVecPerWarp = 2;
constexpr int kVecPerBlock = 8 * kVecPerWarp;  // 8 warps

// The 8 E4M3 codes of one lane's 8 values (two words), all divided by s.
__device__ __forceinline__ uint2 encode8(const uint32_t (&w)[4], float s) {
  uint32_t packed[2] = {0u, 0u};
  if (s >= kFastQuotientMinScale) {
    const float r = __frcp_rn(s);
    const uint64_t neg_s2 = ptx::f32x2(-s, -s), r2 = ptx::f32x2(r, r);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      // BF16 -> FP32 is exact: the BF16 bits are the top half.
      const uint64_t x2 = ptx::f32x2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
      float q0, q1;
      ptx::f32x2_split(quotient_rn_x2(x2, neg_s2, r2), q0, q1);
      packed[i >> 1] |= static_cast<uint32_t>(ptx::cvt_e4m3x2(q0, q1)) << (16 * (i & 1));
    }
  } else if (s > 0.0f) {  // scales below 2^-100: the IEEE division
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t pair = ptx::cvt_e4m3x2(__fdiv_rn(__uint_as_float(w[i] << 16), s),
                                            __fdiv_rn(__uint_as_float(w[i] & 0xffff0000u), s));
      packed[i >> 1] |= pair << (16 * (i & 1));
    }
  }
  return make_uint2(packed[0], packed[1]);
}

// Scale of vector vec = (row, head): [row][heads], or head-major [head][stride]
// where a batch's sequence b starts at column col_begin[b] (a multiple of 4).
__device__ __forceinline__ void store_scale(float* scale, int vec, float s, int heads,
                                            int scale_stride, int head_major,
                                            const ScaleColumns& cols) {
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

__global__ void __launch_bounds__(256)
    quantize_fp8_kernel(const __nv_bfloat16* __restrict__ x, uint8_t* __restrict__ codes,
                        float* __restrict__ scale, int n_vec, int heads, int scale_stride,
                        int head_major, const __grid_constant__ ScaleColumns cols) {
  const int lane = threadIdx.x & 31;
  const int n_task = (n_vec + kVecPerWarp - 1) / kVecPerWarp;  // task t: vectors t*2, t*2+1
  const int stride = static_cast<int>(gridDim.x) * 8;
  // This lane's 16 bytes of the vectors of task t (zeros past the end).
  auto load = [&](int t, uint4 (&raw)[kVecPerWarp]) {
#pragma unroll
    for (int u = 0; u < kVecPerWarp; ++u) {
      const int vec = t * kVecPerWarp + u;
      raw[u] = vec < n_vec
                   ? reinterpret_cast<const uint4*>(x + static_cast<size_t>(vec) * kHeadDim)[lane]
                   : make_uint4(0, 0, 0, 0);
    }
  };
  int t = static_cast<int>(blockIdx.x) * 8 + static_cast<int>(threadIdx.x >> 5);
  uint4 cur[kVecPerWarp];
  load(t, cur);
  for (; t < n_task; t += stride) {  // warp-uniform
    uint4 nxt[kVecPerWarp];
    load(t + stride, nxt);
#pragma unroll
    for (int u = 0; u < kVecPerWarp; ++u) {
      const int vec = t * kVecPerWarp + u;
      if (vec >= n_vec) break;  // warp-uniform
      const uint32_t w[4] = {cur[u].x, cur[u].y, cur[u].z, cur[u].w};
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        amax = ptx::fmax3(amax, fabsf(__uint_as_float(w[i] << 16)),
                          fabsf(__uint_as_float(w[i] & 0xffff0000u)));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const float s = __fdiv_rn(amax, kE4m3Max);
      reinterpret_cast<uint2*>(codes + static_cast<size_t>(vec) * kHeadDim)[lane] = encode8(w, s);
      if (lane == 0) store_scale(scale, vec, s, heads, scale_stride, head_major, cols);
    }
#pragma unroll
    for (int u = 0; u < kVecPerWarp; ++u) cur[u] = nxt[u];
  }
}

// Per-channel quantisation of V for the quantised PV (same report's final
// submission multiplies P by V in 8 bits; the scaling is not given). Reading:
// channel c of KV head g over all kv_len keys is one vector, with s = max_j
// |v[j][g][c]| / 448 and codes E4M3(v / s) under the rounding rules above. The
// codes are stored transposed, [g][c][key] with a row stride of v_stride
// bytes, so that a 128-key tile of V is a K-major operand (one 128-byte row of
// keys per channel) for the kind::f8f6f4 MMA; the scale multiplies column c of
// P.V after the product.
//
// Three passes: (1) amax: block b reduces keys [b*kAmaxKeys, ...) for all 1024
// (head, channel) pairs, a thread per 4 channels (8 bytes of each key row:
// coalesced 2 KB rows), then one atomicMax on the float bits per channel (|v|
// >= 0, so the bits order like the values) into v_scale, cleared before;
// (2) encode: a block per (128 keys, 32 channels) tile takes its 32 channels'
// s = amax / 448 and RN(1 / s) into shared memory once, reads the tile's key
// rows (64 bytes each), forms the quotients (fp8_quotient.cuh) and writes 32
// channel rows of 128 codes through shared memory; (3) v_scale = amax / 448
// in place.
constexpr int kAmaxKeys = 64;

__global__ void __launch_bounds__(256) v_amax_kernel(const __nv_bfloat16* __restrict__ v,
                                                     unsigned int* __restrict__ amax_bits,
                                                     int kv_len) {
  const int c4 = threadIdx.x;  // channels 4*c4 .. 4*c4+3 of the 1024 (head-major)
  const int k0 = blockIdx.x * kAmaxKeys, k1 = min(kv_len, k0 + kAmaxKeys);
  float m[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int j0 = k0; j0 < k1; j0 += 8) {  // eight independent loads in flight per thread
    uint2 raw[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      raw[u] = j0 + u < k1
                   ? reinterpret_cast<const uint2*>(v + static_cast<size_t>(j0 + u) * kKvHeads * kHeadDim)[c4]
                   : make_uint2(0, 0);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      m[0] = fmaxf(m[0], fabsf(__uint_as_float(raw[u].x << 16)));
      m[1] = fmaxf(m[1], fabsf(__uint_as_float(raw[u].x & 0xffff0000u)));
      m[2] = fmaxf(m[2], fabsf(__uint_as_float(raw[u].y << 16)));
      m[3] = fmaxf(m[3], fabsf(__uint_as_float(raw[u].y & 0xffff0000u)));
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) atomicMax(amax_bits + 4 * c4 + i, __float_as_uint(m[i]));
}

__global__ void __launch_bounds__(256) v_encode_kernel(const __nv_bfloat16* __restrict__ v,
                                                       const unsigned int* __restrict__ amax_bits,
                                                       uint8_t* __restrict__ codes, int kv_len,
                                                       int v_stride) {
  __shared__ uint8_t tile[32][128 + 16];  // [channel][key], rows padded against bank conflicts
  __shared__ float ch_s[32], ch_r[32];    // per channel: s and RN(1 / s) (0 below the fast range)
  const int key0 = blockIdx.x * 128;
  const int ch0 = blockIdx.y * 32;  // of the 1024 (head, channel) pairs
  const int t = threadIdx.x;
  if (t < 32) {
    const float s = __fdiv_rn(__uint_as_float(amax_bits[ch0 + t]), kE4m3Max);
    ch_s[t] = s;
    ch_r[t] = s >= kFastQuotientMinScale ? __frcp_rn(s) : 0.0f;
  }
  __syncthreads();
  // Read: 128 key rows of 32 channels (64 bytes): thread t takes key t/2, channels
  // 16*(t%2) .. +15, for keys key0 .. key0+127.
  const int kr = t >> 1, half = t & 1;
  const int key = key0 + kr;
  if (key < kv_len) {
    const uint4* src = reinterpret_cast<const uint4*>(
        v + static_cast<size_t>(key) * kKvHeads * kHeadDim + ch0 + 16 * half);
    const uint4 a = src[0], b = src[1];
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = 16 * half + 2 * i;  // channels c, c + 1
      const float x0 = __uint_as_float(w[i] << 16), x1 = __uint_as_float(w[i] & 0xffff0000u);
      const float s0 = ch_s[c], s1 = ch_s[c + 1];
      float q0, q1;
      if (ch_r[c] != 0.0f && ch_r[c + 1] != 0.0f) {
        ptx::f32x2_split(quotient_rn_x2(ptx::f32x2(x0, x1), ptx::f32x2(-s0, -s1),
                                        ptx::f32x2(ch_r[c], ch_r[c + 1])), q0, q1);
      } else {  // a channel whose scale is 0 or below 2^-100
        q0 = s0 > 0.0f ? __fdiv_rn(x0, s0) : 0.0f;
        q1 = s1 > 0.0f ? __fdiv_rn(x1, s1) : 0.0f;
      }
      const uint32_t pair = ptx::cvt_e4m3x2(q0, q1);
      tile[c][kr] = static_cast<uint8_t>(pair & 0xffu);
      tile[c + 1][kr] = static_cast<uint8_t>(pair >> 8);
    }
  }
  __syncthreads();
  // Write: 32 channel rows of up to 128 codes; thread t: channel t/8, 16 keys.
  const int c = t >> 3, part = t & 7;
  const int g = (ch0 + c) / kHeadDim, d = (ch0 + c) % kHeadDim;
  const int kk = key0 + 16 * part;
  if (kk < kv_len) {
    uint8_t* dst = codes + (static_cast<size_t>(g) * kHeadDim + d) * v_stride + kk;
    if (kk + 16 <= kv_len) {
      *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(&tile[c][16 * part]);
    } else {
      for (int i = 0; i < kv_len - kk; ++i) dst[i] = tile[c][16 * part + i];
    }
  }
}

__global__ void v_scale_kernel(float* __restrict__ scale) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < kKvHeads * kHeadDim) scale[i] = __fdiv_rn(scale[i], kE4m3Max);  // amax bits -> s
}

}  // namespace

cudaError_t launch_quantize_v_fp8(const void* v, void* codes, float* scale, int kv_len,
                                  int v_stride, cudaStream_t stream) {
  if (kv_len == 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(scale, 0, kKvHeads * kHeadDim * sizeof(float), stream);
  if (e != cudaSuccess) return e;
  auto* amax = reinterpret_cast<unsigned int*>(scale);
  v_amax_kernel<<<(kv_len + kAmaxKeys - 1) / kAmaxKeys, 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(v), amax, kv_len);
  v_encode_kernel<<<dim3((kv_len + 127) / 128, kKvHeads * kHeadDim / 32), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(v), amax, static_cast<uint8_t*>(codes), kv_len, v_stride);
  v_scale_kernel<<<(kKvHeads * kHeadDim + 255) / 256, 256, 0, stream>>>(scale);
  return cudaGetLastError();
}

cudaError_t launch_quantize_fp8(const void* x, void* codes, float* scale, int rows, int heads,
                                int scale_stride, bool head_major, const ScaleColumns& cols,
                                int num_sms, cudaStream_t stream) {
  const int n_vec = rows * heads;
  if (n_vec == 0) return cudaSuccess;
  // Persistent: at most 8 blocks per SM (what fits), each warp looping over tasks.
  const int blocks = std::min((n_vec + kVecPerBlock - 1) / kVecPerBlock, 8 * std::max(num_sms, 1));
  quantize_fp8_kernel<<<blocks, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(x),
                                                   static_cast<uint8_t*>(codes), scale, n_vec,
                                                   heads, scale_stride, head_major ? 1 : 0, cols);
  return cudaGetLastError();
}

}  // namespace gqa
