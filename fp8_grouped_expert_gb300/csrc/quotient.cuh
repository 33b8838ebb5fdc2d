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
// sign.  Outside that range of s the callers divide.  A NaN x gives NaN either way, and an
// infinite x makes the caller's amax infinite and its s out of the range (the outputs for
// non-finite inputs are meaningless; the quantizers report them).  cast8 below is the
// 8-value cast every e4m3 activation quantizer shares.
#pragma once

#include "fge_device.cuh"

namespace fge {

__device__ __forceinline__ bool quot_fast_ok(float s) {
  return s >= 0x1p-90f && s <= 0x1p+120f;  // false for inf and NaN
}

__device__ __forceinline__ float quot_rn(float x, float s, float y) {
  const float q0 = __fmul_rn(x, y);
  const float r = -__fmaf_rn(q0, s, -x);
  return __fmaf_rn(r, y, q0);
}

// The e4m3 codes of 8 bf16 values divided by s (the IEEE quotient, then round to nearest
// even).  y = RN(1/s) and fast = quot_fast_ok(s), both from the caller: the quotient comes
// from the reciprocal (quotient.cuh) when s is in that method's range, else by division.
// A NaN value gives a NaN quotient either way.
__device__ __forceinline__ uint2 cast8(const uint4& v, float s, float y, bool fast) {
  const float f[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                      bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
  float d[8];
  if (fast) {
#pragma unroll
    for (int i = 0; i < 8; ++i) d[i] = quot_rn(f[i], s, y);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) d[i] = __fdiv_rn(f[i], s);
  }
  uint2 q;
  q.x = cvt_e4m3x4(d[0], d[1], d[2], d[3]);
  q.y = cvt_e4m3x4(d[4], d[5], d[6], d[7]);
  return q;
}

}  // namespace fge
