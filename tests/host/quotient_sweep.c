/* Host check of the quantizers' quotient: for x with an 8-bit significand (a bfloat16
 * value) and s with a 24-bit significand, y = RN(1/s), q0 = RN(x y), r = -(q0 s - x) by
 * one fused multiply-add, q1 = RN(q0 + r y) must equal the IEEE quotient RN(x / s).
 * Scaling x and s by powers of two scales every step exactly while nothing leaves the
 * normal range, so significands in [1, 2) cover every normal case.
 * Usage: quotient_sweep STRIDE [plain]   (every STRIDE-th significand of s; "plain" checks
 * q0 instead of q1 and must find mismatches).  Prints "pairs N mismatches M". */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static float from_bits(uint32_t u) {
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

int main(int argc, char** argv) {
  const uint32_t stride = argc > 1 ? (uint32_t)strtoul(argv[1], NULL, 10) : 1u;
  const int plain = argc > 2 && strcmp(argv[2], "plain") == 0;
  long long pairs = 0, bad = 0;
  for (uint32_t xm = 0; xm < 128u; ++xm) {
    const float x = from_bits((127u << 23) | (xm << 16));
    for (uint32_t sm = 0; sm < (1u << 23); sm += stride) {
      const float s = from_bits((127u << 23) | sm);
      const float y = 1.0f / s;
      const float q0 = x * y;
      const float r = -fmaf(q0, s, -x);
      const float q1 = plain ? q0 : fmaf(r, y, q0);
      ++pairs;
      if (q1 != x / s) ++bad;
    }
  }
  printf("pairs %lld mismatches %lld\n", pairs, bad);
  return 0;
}
