/* Host check of the quantizers' quotient across exponents and signs, in the two domains the
 * kernels can meet.  Mode "amax": the scale is derived as the kernels derive it,
 * s = max(RN(amax / 448), 2^-126) for a random bfloat16 amax > 0 of any exponent, and x is
 * any bfloat16 value with |x| <= amax (zeros, subnormals, both signs), so |x / s| stays near
 * or below 448.  Mode "wide": s is any float in [2^-90, 2^120] and x any bfloat16 value with
 * |x / s| < 2^126.  Only pairs with s in [2^-90, 2^120] (where the kernels take the
 * reciprocal path) are counted.  A pair agrees when the corrected quotient has the sign of
 * the IEEE quotient and either equals it or both lie below 2^-10, where every value rounds
 * to an e4m3 zero; so agreement means equal e4m3 codes.  (Below |x| ~ 2^-103 the residual
 * x - q0 s is no longer exact and the two may differ in the last place, always below 2^-10.)
 * Mode "scale" is exhaustive instead: the group scale max(RN(amax / 448), 2^-126) taken by
 * the same correction step from the constant RN(1/448) must equal the one from the division
 * for every finite bfloat16 amax (COUNT and SEED are ignored).
 * Usage: quotient_range COUNT SEED amax|wide|scale.  Prints "pairs N mismatches M". */
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

static uint64_t state;
static uint32_t next_u32(void) { /* xorshift64* */
  state ^= state >> 12;
  state ^= state << 25;
  state ^= state >> 27;
  return (uint32_t)((state * 2685821657736338717ULL) >> 32);
}

static float random_bf16(void) { return from_bits((next_u32() & 0xFFFFu) << 16); }

int main(int argc, char** argv) {
  const long long n = argc > 1 ? atoll(argv[1]) : 1000000;
  state = (argc > 2 ? strtoull(argv[2], NULL, 10) : 1) * 2654435761ULL + 1;
  const int wide = argc > 3 && strcmp(argv[3], "wide") == 0;
  long long bad = 0, pairs = 0;
  if (argc > 3 && strcmp(argv[3], "scale") == 0) {
    const float y448 = 0x1.24924ap-9f;
    if (y448 != 1.0f / 448.0f) bad = 1; /* the constant is RN(1/448) */
    for (uint32_t h = 0; h < 0x7F80u; ++h) {
      const float amax = from_bits(h << 16);
      const float q0 = amax * y448;
      const float r = -fmaf(q0, 448.0f, -amax);
      float s_fast = fmaf(r, y448, q0);
      float s_div = amax / 448.0f;
      if (amax == 0.0f) s_fast = s_div = 1.0f;
      if (s_fast < 0x1p-126f) s_fast = 0x1p-126f;
      if (s_div < 0x1p-126f) s_div = 0x1p-126f;
      ++pairs;
      if (s_fast != s_div) ++bad;
    }
    printf("pairs %lld mismatches %lld\n", pairs, bad);
    return 0;
  }
  while (pairs < n) {
    float x, s;
    if (wide) {
      const int es = (int)(next_u32() % 211u) - 90;
      s = ldexpf(1.0f + (float)(next_u32() & 0x7FFFFFu) / 8388608.0f, es);
      x = random_bf16();
      if (!isfinite(x) || !(fabsf(x / s) < 0x1p126f)) continue;
    } else {
      const float amax = fabsf(random_bf16());
      if (!isfinite(amax) || amax == 0.0f) continue;
      s = amax / 448.0f;
      if (s < 0x1p-126f) s = 0x1p-126f;
      /* x: a random bfloat16 pattern no larger in magnitude than amax, its exponent drawn
       * at most that of amax so that every binade below amax is reached */
      uint32_t amax_bits;
      memcpy(&amax_bits, &amax, sizeof amax_bits);
      const uint32_t top = amax_bits >> 16; /* bf16 pattern of amax */
      const uint32_t mag = next_u32() % (top + 1u);
      x = from_bits(((next_u32() & 1u) << 31) | (mag << 16));
    }
    if (s < 0x1p-90f || s > 0x1p+120f) continue;
    ++pairs;
    const float y = 1.0f / s;
    const float q0 = x * y;
    const float r = -fmaf(q0, s, -x);
    const float q1 = fmaf(r, y, q0);
    const float q = x / s;
    const int agree = signbit(q1) == signbit(q) &&
                      (q1 == q || (fabsf(q1) < 0x1p-10f && fabsf(q) < 0x1p-10f));
    if (!agree) ++bad;
  }
  printf("pairs %lld mismatches %lld\n", pairs, bad);
  return 0;
}
