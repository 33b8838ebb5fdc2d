// The IEEE round-to-nearest quotient x / s of the activation quantizers, from one correctly
// rounded reciprocal per scale.  With y = RN(1/s), q0 = RN(x y) and the exact residual
// r = x - q0 s (one FMA), RN(q0 + r y) is the correctly rounded quotient (Markstein's
// correction step, "Computation of elementary functions on the IBM RISC System/6000
// processor", 1990).  For the inputs here -- x a bfloat16 value (at most 8 significant
// bits), s a normal float in [2^-90, 2^120] -- that holds for every pair of significands
// (all 2^7 x 2^23 of them checked against the division on the host, tests/host), and
// scaling both by powers of two keeps it while the steps stay normal.  Below |x| ~ 2^-103 the
// residual is subnormal and inexact and the result may be off by one unit in the last place,
// but then |x / s| < 2^-13 and both round to the same signed e4m3 zero; the quotient must not
// overflow (q0 would be infinite and the result NaN), which the callers guarantee by deriving
// s = amax / 448 from the values they cast.  Both corners are sampled on the host across all
// exponents and signs.  The residual is formed as -(q0 s - x) so that a zero x keeps its
// sign.  Outside that range of s, or for a non-finite x, the callers divide.
#pragma once

namespace fge {

__device__ __forceinline__ bool quot_fast_ok(float s) {
  return s >= 0x1p-90f && s <= 0x1p+120f;  // false for inf and NaN
}

__device__ __forceinline__ float quot_rn(float x, float s, float y) {
  const float q0 = __fmul_rn(x, y);
  const float r = -__fmaf_rn(q0, s, -x);
  return __fmaf_rn(r, y, q0);
}

}  // namespace fge
