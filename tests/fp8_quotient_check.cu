// Exhaustive check of the FP8 quantisers' division-free quotient
// (gqa_chunked_prefill_gb300/csrc/fp8_quotient.cuh) against CUDA's IEEE
// round-to-nearest division, over every pair the quantisers can meet: x any
// finite BF16 value, m any positive finite BF16 maximum with |x| <= m, and
// s = RN(m / 448) at or above the fast path's smallest scale. Prints the number
// of pairs checked, of E4M3 codes that differ, of FP32 quotients that differ,
// and of those where either quotient is 2^-11 or more in magnitude (below that
// E4M3 rounds both to a zero of x's sign: its smallest step is 2^-9); exits 0.
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>

#include "fp8_quotient.cuh"

namespace {

__global__ void check_kernel(unsigned long long* counts, unsigned int* first) {
  __shared__ unsigned long long block_counts[4];
  if (threadIdx.x < 4) block_counts[threadIdx.x] = 0;
  __syncthreads();
  const uint32_t m_bits = 1u + blockIdx.x;  // 0x0001 .. 0x7F7F
  const float m = __uint_as_float(m_bits << 16);
  const float s = __fdiv_rn(m, 448.0f);
  unsigned long long n = 0, bad_q = 0, bad_code = 0, bad_q_range = 0;
  if (s >= gqa::kFastQuotientMinScale) {
    const float r = __frcp_rn(s);
    const uint64_t neg_s2 = gqa::ptx::f32x2(-s, -s), r2 = gqa::ptx::f32x2(r, r);
    for (uint32_t xb = threadIdx.x; xb < 65536u; xb += blockDim.x) {
      if ((xb & 0x7fffu) > m_bits) continue;  // |x| > m (and every NaN / Inf, as m is finite)
      const float x = __uint_as_float(xb << 16);
      const float ref = __fdiv_rn(x, s);
      float q, unused;
      gqa::ptx::f32x2_split(gqa::quotient_rn_x2(gqa::ptx::f32x2(x, x), neg_s2, r2), q, unused);
      ++n;
      if (__float_as_uint(q) != __float_as_uint(ref)) {
        ++bad_q;
        if (fmaxf(fabsf(q), fabsf(ref)) >= 4.8828125e-4f) {  // 2^-11
          ++bad_q_range;
          atomicCAS(first, 0u, (m_bits << 16) | xb);
        }
      }
      if ((gqa::ptx::cvt_e4m3x2(q, 0.0f) & 0xffu) != (gqa::ptx::cvt_e4m3x2(ref, 0.0f) & 0xffu))
        ++bad_code;
    }
  }
  atomicAdd(&block_counts[0], n);
  atomicAdd(&block_counts[1], bad_q);
  atomicAdd(&block_counts[2], bad_code);
  atomicAdd(&block_counts[3], bad_q_range);
  __syncthreads();
  if (threadIdx.x < 4) atomicAdd(counts + threadIdx.x, block_counts[threadIdx.x]);
}

}  // namespace

int main() {
  unsigned long long* counts = nullptr;
  unsigned int* first = nullptr;
  if (cudaMalloc(&counts, 4 * sizeof(unsigned long long)) != cudaSuccess ||
      cudaMalloc(&first, sizeof(unsigned int)) != cudaSuccess) {
    std::printf("error cudaMalloc\n");
    return 1;
  }
  cudaMemset(counts, 0, 4 * sizeof(unsigned long long));
  cudaMemset(first, 0, sizeof(unsigned int));
  check_kernel<<<0x7F7F, 256>>>(counts, first);
  unsigned long long h[4] = {0, 0, 0, 0};
  unsigned int hf = 0;
  const cudaError_t e = cudaDeviceSynchronize();
  cudaMemcpy(h, counts, sizeof(h), cudaMemcpyDeviceToHost);
  cudaMemcpy(&hf, first, sizeof(hf), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) {
    std::printf("error %s\n", cudaGetErrorString(e));
    return 1;
  }
  std::printf("checked %llu code_mismatch %llu fp32_mismatch %llu fp32_mismatch_from_2^-11 %llu first 0x%08x\n",
              h[0], h[2], h[1], h[3], hf);
  return 0;
}
