// The quotient x / s of the FP8 quantisers without a division per value.
//
// The quantisers define a code as E4M3(RN(x / s)): the FP32 quotient rounded
// to nearest, then rounded once more to E4M3. With r = RN(1 / s) computed once
// per vector (or per channel), each quotient is
//
//   q0 = RN(x r),  e = x - q0 s (one FMA: exact),  q = RN(q0 + e r),
//
// Markstein's correction ("Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990): q0 is within an ulp of
// x / s, the remainder of such a q0 is a floating-point number, and one fused
// step from it with the correctly rounded reciprocal gives the correctly
// rounded quotient. Two values go through each packed FP32 instruction.
//
// Domain: the quantisers call it only for s >= 2^-100 (normal, with 1 / s far
// from overflow; smaller scales take the IEEE division). The sign is copied
// from x, so that x = -0 gives -0 as the division does. For every BF16 x and
// every BF16 maximum m >= |x| (s = RN(m / 448)) the E4M3 code of the result
// equals that of the IEEE division, and so does the FP32 quotient wherever
// either is 2^-11 or more; below that, a subnormal x leaves the remainder
// inexact and low bits may differ, but E4M3 (smallest step 2^-9) rounds both
// to a zero of x's sign. The GPU test suite checks all ~1.04e9 such pairs.
#pragma once

#include <cstdint>

#include "sm100_ptx.cuh"

namespace gqa {

// Smallest scale the fast quotient is used for.
constexpr float kFastQuotientMinScale = 7.88860905e-31f;  // 2^-100

// RN(x / s) for the pair (x.lo, x.hi) against the pair of scales (s.lo, s.hi),
// given neg_s = (-s.lo, -s.hi) and r = (RN(1 / s.lo), RN(1 / s.hi)).
__device__ __forceinline__ uint64_t quotient_rn_x2(uint64_t x, uint64_t neg_s, uint64_t r) {
  const uint64_t q0 = ptx::mul_f32x2(x, r);
  const uint64_t e = ptx::fma_f32x2(q0, neg_s, x);
  const uint64_t q = ptx::fma_f32x2(e, r, q0);
  constexpr uint64_t kSign = 0x8000000080000000ull;
  return (q & ~kSign) | (x & kSign);
}

}  // namespace gqa
