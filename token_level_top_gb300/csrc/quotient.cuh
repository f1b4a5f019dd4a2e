// quotient.cuh -- a correctly rounded fp32 quotient by FMA, for the quantisers
// (many elements divided by one block or row scale).
#pragma once

#include <math.h>

namespace moe {

// x / den rounded to nearest even (den > 0), from y = 1/den rounded to nearest
// even: q0 = x y, then twice q <- q + (x - q den) y, each remainder taken with one
// FMA.  This is Markstein's correction step (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res. Dev.
// 34(1), 1990): when y is within half an ulp of 1/den and q within one ulp of
// x / den, the remainder is exact and q + r y rounds to the correctly rounded
// quotient.  q0 may miss that by up to half an ulp; the first step brings it
// within one ulp, the second gives the quotient.  The remainder is exact while
// |x| >= 2^-103 or so; callers take this path for den >= kFmaDivMin = 2^-92, where
// every quotient at or above 2^-10 (the smallest e4m3 rounding boundary) has such
// an x, and a smaller quotient one ulp off changes no e4m3 or e2m1 code.  The
// sign of the quotient is that of x, zeros included.
constexpr float kFmaDivMin = 0x1p-92f;

__device__ __forceinline__ float div_by(float x, float den, float y)
{
    float q = __fmul_rn(x, y);
    q = __fmaf_rn(__fmaf_rn(-q, den, x), y, q);
    q = __fmaf_rn(__fmaf_rn(-q, den, x), y, q);
    return copysignf(q, x);
}

}  // namespace moe
