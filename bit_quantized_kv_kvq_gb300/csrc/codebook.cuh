// Quotient of two fp16 values in fp32 for the codebook quantizer, without a
// division: with r = RN(1/s), y0 = RN(x r) is within one ulp of x / s, the
// residual x - y0 s is exact in an fma, and one correction
// y = RN(y0 + (x - y0 s) r) gives the correctly rounded x / s (Markstein's
// division correction, P. Markstein, "Computation of elementary functions on
// the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990).
// kvq_selftest_codebook_quotient checks it against IEEE division for every
// finite fp16 x and every positive finite fp16 s; a zero of either sign may
// come out as +0.
#pragma once

#include <cuda_fp16.h>

namespace kvq {
namespace cb {

__device__ __forceinline__ float quotient(float x, float s, float r) {
  const float y0 = __fmul_rn(x, r);
  const float rem = __fmaf_rn(-y0, s, x);
  return __fmaf_rn(rem, r, y0);
}

}  // namespace cb
}  // namespace kvq
