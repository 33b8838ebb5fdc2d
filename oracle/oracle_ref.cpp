// CPU oracle, single-threaded C++ restatement of the W4A8 grouped-expert MoE prefill path.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product library links or calls this file: only
// the test suite, the smoke check and the cpu_baseline / reference legs of the benchmark do.
// It shares no code, header or table with the CUDA library; inputs reach it as plain arrays.
//
// What it computes is the definition of each step of "FP8 grouped-expert prefill with
// on-chip int4-to-e4m3 dequant" (section 1) and of the dense per-tensor W8A8 projection of
// "feat(qwen4_exp): load-time per-tensor FP8 dense projections" (section "What this adds"),
// with float64 accumulation and plain loops: no blocking, no reordering, no threads.  The
// readings taken where the pages are silent are the same as the numpy restatement in this
// package (the e4m3 variant, the zero-scale floor, the int4 nibble order, top-k ties, the
// gate_up halves, SwiGLU), and each is repeated beside the code that takes it.
//
// The algorithms differ on purpose from the numpy restatement where a rule can be written
// two ways (the e4m3 and bf16 roundings work on the float bits here, on frexp/rint there;
// top-k selects by repeated maximum here, by a sort there), so that the two pin each other.
//
// Build: g++ -O2 -std=c++17 -ffp-contract=off -shared -fPIC.  Contraction stays off so that
// every float64 product and sum is rounded on its own, in the order written.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

constexpr int kGroup = 128;  // K group of the activation and weight scales

// ------------------------------------------------------------------------ e4m3 codec
// OCP E4M3FN: 1 sign, 4 exponent, 3 mantissa bits ("FP8 vs INT4 KV Cache", section "FP8
// (E4M3) vs. Grouped INT4", item 1).  Reading: bias 7, subnormals at exponent field 0, no
// infinities, S.1111.111 is NaN, so the largest finite magnitude is 448 -- the divisor of
// the amax/448 scale on "Module fp8_ffi".
double e4m3_value(uint8_t code) {
  const int e = (code >> 3) & 0xF;
  const int m = code & 0x7;
  if (e == 0xF && m == 0x7) return std::nan("");
  const double mag = e == 0 ? std::ldexp(static_cast<double>(m), -9)
                            : std::ldexp(static_cast<double>(8 + m), e - 10);
  return (code & 0x80) ? -mag : mag;
}

// float32 -> e4m3 code, round to nearest (ties to even) on the exact float value, saturating
// at +-448, sign kept (-0 -> 0x80).  Worked on the float's bits: |x| = m * 2^ex with an
// integer significand m; the e4m3 quantum of [2^E, 2^(E+1)) is 2^(E-3), and 2^-9 below 2^-6.
uint8_t e4m3_code(float x) {
  uint32_t b;
  std::memcpy(&b, &x, 4);
  const uint8_t sign = static_cast<uint8_t>((b >> 31) << 7);
  const uint32_t a = b & 0x7FFFFFFFu;
  if (a > 0x7F800000u) return sign | 0x7F;   // NaN in, NaN out (not used by the path)
  if (a == 0x7F800000u) return sign | 0x7E;  // infinities saturate like large values
  const int ef = static_cast<int>(a >> 23);
  uint32_t m = a & 0x7FFFFFu;
  int ex;
  if (ef == 0) {
    ex = -149;
  } else {
    m |= 0x800000u;
    ex = ef - 150;
  }
  if (m == 0) return sign;
  int msb = 0;
  while ((m >> (msb + 1)) != 0) ++msb;
  const int E = ex + msb;                    // |x| in [2^E, 2^(E+1))
  const int qexp = (E < -6 ? -6 : E) - 3;    // exponent of the quantum
  const int shift = qexp - ex;               // >= 0 except far above the e4m3 range
  uint64_t r;                                // |x| rounded, in quanta
  if (shift <= 0) {
    if (E > 8) return sign | 0x7E;
    r = static_cast<uint64_t>(m) << (-shift);
  } else if (shift > 40) {
    r = 0;
  } else {
    const uint64_t mm = m;
    const uint64_t q = mm >> shift;
    const uint64_t rem = mm & ((uint64_t{1} << shift) - 1);
    const uint64_t half = uint64_t{1} << (shift - 1);
    r = (rem > half || (rem == half && (q & 1))) ? q + 1 : q;
  }
  // value = r * 2^qexp
  if (qexp == -9) {                          // subnormal quantum: r in [0, 8]
    return sign | static_cast<uint8_t>(r);   // r == 8 is 2^-6, code 0x08, the smallest normal
  }
  int Eo = qexp + 3;                         // r in [8, 16]
  if (r == 16) {
    r = 8;
    ++Eo;
  }
  if (Eo > 8 || (Eo == 8 && r > 14)) return sign | 0x7E;  // above 448: saturate
  return sign | static_cast<uint8_t>(((Eo + 7) << 3) | static_cast<int>(r - 8));
}

// float64 -> bfloat16 bits, one rounding (nearest, ties to even), worked on the double's
// bits.  bfloat16 keeps 8 significant bits; below 2^-126 its quantum is 2^-133.  Finite
// inputs whose magnitude stays below 2^128.
uint16_t bf16_bits(double v) {
  uint64_t b;
  std::memcpy(&b, &v, 8);
  const uint16_t sign = static_cast<uint16_t>((b >> 63) << 15);
  const uint64_t a = b & 0x7FFFFFFFFFFFFFFFull;
  const int ef = static_cast<int>(a >> 52);
  uint64_t m = a & 0xFFFFFFFFFFFFFull;
  int ex;
  if (ef == 0) {
    ex = -1074;
  } else {
    m |= 0x10000000000000ull;
    ex = ef - 1075;
  }
  if (m == 0) return sign;
  int msb = 0;
  while ((m >> (msb + 1)) != 0) ++msb;
  const int E = ex + msb;
  const int qexp = (E < -126 ? -126 : E) - 7;
  const int shift = qexp - ex;
  uint64_t r;
  if (shift <= 0) {
    r = m << (-shift);
  } else if (shift > 60) {
    r = 0;
  } else {
    const uint64_t q = m >> shift;
    const uint64_t rem = m & ((uint64_t{1} << shift) - 1);
    const uint64_t half = uint64_t{1} << (shift - 1);
    r = (rem > half || (rem == half && (q & 1))) ? q + 1 : q;
  }
  if (qexp == -133) {                        // subnormal: r in [0, 128]; 128 is 2^-126
    return sign | static_cast<uint16_t>(r);
  }
  int Eo = qexp + 7;                         // r in [128, 256]
  if (r == 256) {
    r = 128;
    ++Eo;
  }
  return sign | static_cast<uint16_t>(((Eo + 127) << 7) | static_cast<int>(r - 128));
}

float bf16_to_float(uint16_t h) {
  const uint32_t b = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &b, 4);
  return f;
}

// int4 element kk of a packed row: two's complement nibbles, element 2b in the low nibble
// of byte b ("FP8 grouped-expert prefill ...", section 1: a resident packed-int4 bank, two
// values a byte; the low nibble first follows the unpack snippet of "FP8 vs INT4 KV Cache").
int int4_at(const uint8_t* row, int64_t kk) {
  const uint8_t byte = row[kk >> 1];
  const int nib = (kk & 1) ? (byte >> 4) : (byte & 0xF);
  return nib >= 8 ? nib - 16 : nib;
}

// Scale of a group or tensor: s = fp32(amax / 448) ("Module fp8_ffi": amax/448).  Readings:
// amax == 0 gives s = 1; s below the smallest normal float (2^-126) is raised to 2^-126
// (the zero-input floor of "feat(qwen4_exp) ...", section "Testing", has no printed value).
float scale_from_amax(float amax) {
  if (amax == 0.0f) return 1.0f;
  const float s = amax / 448.0f;
  const float floor_s = 1.1754943508222875e-38f;  // 2^-126
  return s < floor_s ? floor_s : s;
}

// Codes of n values sharing one scale: e4m3(fp32(x / s)), the IEEE float quotient first.
void quant_run(const float* x, int64_t n, float s, uint8_t* q) {
  for (int64_t i = 0; i < n; ++i) q[i] = e4m3_code(x[i] / s);
}

float amax_of(const float* x, int64_t n) {
  float a = 0.0f;
  for (int64_t i = 0; i < n; ++i) a = std::fabs(x[i]) > a ? std::fabs(x[i]) : a;
  return a;
}

}  // namespace

extern "C" {

double fo_e4m3_decode(uint8_t code) { return e4m3_value(code); }
uint8_t fo_e4m3_encode(float x) { return e4m3_code(x); }

void fo_e4m3_encode_n(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_code(x[i]);
}

void fo_bf16_round_n(const double* v, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = bf16_bits(v[i]);
}

// Exhaustive check of the encoder on every float32 whose magnitude lies in [2^lo, 2^hi),
// both signs, against a brute-force search of the 127 finite magnitudes for the nearest one
// (ties to the even code), 448 above the range.  Returns the number of mismatches.
int64_t fo_e4m3_encode_selfcheck(int lo, int hi) {
  double mags[127];
  for (int c = 0; c < 127; ++c) mags[c] = e4m3_value(static_cast<uint8_t>(c));
  int64_t bad = 0;
  const uint32_t first = static_cast<uint32_t>(lo + 127) << 23;
  const uint32_t last = static_cast<uint32_t>(hi + 127) << 23;
  for (uint32_t bits = first; bits < last; ++bits) {
    float f;
    std::memcpy(&f, &bits, 4);
    const double v = f;
    // binary search for the first magnitude >= v, then compare with its neighbour below
    int lo_i = 0, hi_i = 126;
    if (v >= mags[126]) {
      lo_i = hi_i = 126;
    } else {
      while (lo_i < hi_i) {
        const int mid = (lo_i + hi_i) / 2;
        if (mags[mid] >= v) hi_i = mid; else lo_i = mid + 1;
      }
    }
    int want = lo_i;
    if (lo_i > 0 && v < mags[126]) {
      const double dlo = v - mags[lo_i - 1], dhi = mags[lo_i] - v;
      if (dlo < dhi || (dlo == dhi && ((lo_i - 1) % 2 == 0))) want = lo_i - 1;
    }
    const uint8_t got_pos = e4m3_code(f);
    const uint8_t got_neg = e4m3_code(-f);
    if (got_pos != want) ++bad;
    if (got_neg != (0x80 | want)) ++bad;
  }
  return bad;
}

// Activation quantization per (row, 128-K group) ("FP8 grouped-expert prefill ...",
// section 1): amax over the group, s = fp32(amax/448), q = e4m3(fp32(x/s)).
// x float [M, K] (bf16 values widened exactly); q [M, K]; s [M, K/128].
void fo_quant_g128(const float* x, int64_t M, int64_t K, uint8_t* q, float* s) {
  const int64_t G = K / kGroup;
  for (int64_t r = 0; r < M; ++r) {
    for (int64_t g = 0; g < G; ++g) {
      const float* xg = x + r * K + g * kGroup;
      const float sg = scale_from_amax(amax_of(xg, kGroup));
      s[r * G + g] = sg;
      quant_run(xg, kGroup, sg, q + r * K + g * kGroup);
    }
  }
}

// Dynamic per-tensor quantization: one amax over all M*K values, then the same cast
// ("feat(qwen4_exp) ...", section "What this adds": amax pass, then the cast).
void fo_quant_per_tensor(const float* x, int64_t M, int64_t K, uint8_t* q, float* s) {
  const float sg = scale_from_amax(amax_of(x, M * K));
  *s = sg;
  quant_run(x, M * K, sg, q);
}

// One scale per row (the row-wise alternative of "feat(qwen4_exp) ...", section "Limits").
void fo_quant_per_row(const float* x, int64_t M, int64_t K, uint8_t* q, float* s) {
  for (int64_t r = 0; r < M; ++r) {
    s[r] = scale_from_amax(amax_of(x + r * K, K));
    quant_run(x + r * K, K, s[r], q + r * K);
  }
}

// Top-k routing.  Reading (the pages name routed tokens, not the rule): the k largest
// logits, ties toward the lower expert id, picked one at a time; the gates are the softmax
// over the chosen logits, exp(l_j - l_max) / sum exp(l - l_max), in float64, then float32.
void fo_topk_gate(const float* logits, int64_t T, int E, int k, int32_t* ids, float* gates) {
  std::vector<char> taken(E);
  std::vector<double> w(k);
  for (int64_t t = 0; t < T; ++t) {
    const float* l = logits + t * E;
    std::fill(taken.begin(), taken.end(), 0);
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || l[e] > l[best]) best = e;   // strict: the first (lowest) id wins ties
      }
      taken[best] = 1;
      ids[t * k + j] = best;
    }
    const double lmax = l[ids[t * k]];
    double sum = 0.0;
    for (int j = 0; j < k; ++j) {
      w[j] = std::exp(static_cast<double>(l[ids[t * k + j]]) - lmax);
      sum += w[j];
    }
    for (int j = 0; j < k; ++j) gates[t * k + j] = static_cast<float>(w[j] / sum);
  }
}

// Expert-contiguous rows ("FP8 grouped-expert prefill ...", section 1: one grouped GEMM
// over all routed tokens).  counts by expert, offsets = exclusive prefix sum, rows ordered
// by (expert, token, slot) -- a stable counting sort -- and each row copies its token's
// quantized activations and group scales.  aq/as may be null (indices only).
void fo_moe_permute(const int32_t* ids, int64_t T, int k, int E, const uint8_t* xq,
                    const float* xs, int64_t H, int32_t* counts, int32_t* offsets,
                    int32_t* row_token, int32_t* token_row, uint8_t* aq, float* as) {
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t i = 0; i < T * k; ++i) counts[ids[i]] += 1;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  std::vector<int32_t> cursor(offsets, offsets + E);
  const int64_t G = H / kGroup;
  for (int64_t t = 0; t < T; ++t) {
    for (int j = 0; j < k; ++j) {
      const int32_t r = cursor[ids[t * k + j]]++;
      row_token[r] = static_cast<int32_t>(t);
      token_row[t * k + j] = r;
      if (aq) std::memcpy(aq + r * H, xq + t * H, H);
      if (as) std::memcpy(as + r * G, xs + t * G, G * sizeof(float));
    }
  }
}

// The grouped expert GEMM by its definition ("FP8 grouped-expert prefill ...", section 1):
// for expert e and each of its rows r in [offsets[e], offsets[e+1]),
//   C[r, n] = sum_g as[r, g] * sw[e, n, g] * sum_{kk in g} dec(aq[r, kk]) * q[e, n, kk].
// The group sum is exact in float64 (products of at most 7 significant bits, 128 terms);
// the scale product as*sw is exact in float64; the scaled group sums are added in group
// order.  aq [R, K]; as [R, K/128]; w [E, N, K/2]; sw [E, N, K/128]; out float64 [R, N].
void fo_grouped_gemm_w4a8(const uint8_t* aq, const float* as, const int32_t* offsets, int E,
                          const uint8_t* w, const float* sw, int64_t N, int64_t K, int64_t R,
                          double* out) {
  const int64_t G = K / kGroup;
  for (int64_t i = 0; i < R * N; ++i) out[i] = 0.0;
  std::vector<double> arow(K);
  std::vector<double> wq(N * K);
  for (int e = 0; e < E; ++e) {
    const int64_t r0 = offsets[e], r1 = offsets[e + 1];
    if (r1 == r0) continue;
    for (int64_t n = 0; n < N; ++n) {
      const uint8_t* wrow = w + (static_cast<int64_t>(e) * N + n) * (K / 2);
      for (int64_t kk = 0; kk < K; ++kk) wq[n * K + kk] = int4_at(wrow, kk);
    }
    for (int64_t r = r0; r < r1; ++r) {
      for (int64_t kk = 0; kk < K; ++kk) arow[kk] = e4m3_value(aq[r * K + kk]);
      for (int64_t n = 0; n < N; ++n) {
        double acc = 0.0;
        for (int64_t g = 0; g < G; ++g) {
          double part = 0.0;
          for (int64_t kk = g * kGroup; kk < (g + 1) * kGroup; ++kk) part += arow[kk] * wq[n * K + kk];
          const double scale = static_cast<double>(as[r * G + g]) *
                                static_cast<double>(sw[(static_cast<int64_t>(e) * N + n) * G + g]);
          acc += scale * part;
        }
        out[r * N + n] = acc;
      }
    }
  }
}

// SwiGLU between the expert GEMMs, then the per-(row, 128) requantization.  Readings: the
// merged gate_up output holds gate in columns [0, I) and up in [I, 2I); the accumulator is
// float32 on the device, so C is rounded to float32 first; h = fp32(silu(g) * u) with
// silu(g) = g / (1 + exp(-g)) in float64.  c [R, 2I]; hq [R, I]; hs [R, I/128]; h [R, I].
void fo_swiglu_requant(const double* c, int64_t R, int64_t I, uint8_t* hq, float* hs, float* h) {
  for (int64_t r = 0; r < R; ++r) {
    for (int64_t i = 0; i < I; ++i) {
      const double g = static_cast<float>(c[r * 2 * I + i]);
      const double u = static_cast<float>(c[r * 2 * I + I + i]);
      h[r * I + i] = static_cast<float>(g / (1.0 + std::exp(-g)) * u);
    }
  }
  fo_quant_g128(h, R, I, hq, hs);
}

// Gate-weighted sum of each token's k expert rows, in slot order, float64.  Reading (the
// pages do not describe it): out[t] = sum_j gates[t, j] * y[token_row[t, j]].
void fo_moe_combine(const float* y, const int32_t* token_row, const float* gates, int64_t T,
                    int k, int64_t H, double* out) {
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t c = 0; c < H; ++c) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j)
        acc += static_cast<double>(gates[t * k + j]) *
               static_cast<double>(y[static_cast<int64_t>(token_row[t * k + j]) * H + c]);
      out[t * H + c] = acc;
    }
  }
}

// Dense W8A8 GEMM with per-tensor scales ("feat(qwen4_exp) ...", section "What this adds";
// "Module fp8_ffi": one scalar applied to the GEMM): Y = (sa * sw) * sum_k dec(a) dec(w).
// The dot product is exact in float64 for K <= 2^15 (products of 8 significant bits).
void fo_linear_w8a8_gemm(const uint8_t* aq, const float* sa_rows, float sa, const uint8_t* wq,
                         float sw, int64_t M, int64_t N, int64_t K, double* out) {
  std::vector<double> wd(K), ad(K);
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t kk = 0; kk < K; ++kk) wd[kk] = e4m3_value(wq[n * K + kk]);
    for (int64_t m = 0; m < M; ++m) {
      double dot = 0.0;
      for (int64_t kk = 0; kk < K; ++kk) dot += e4m3_value(aq[m * K + kk]) * wd[kk];
      const double s = static_cast<double>(sa_rows ? sa_rows[m] : sa) * static_cast<double>(sw);
      out[m * N + n] = s * dot;
    }
  }
}

// One MoE FFN prefill layer, the stages in the order of "FP8 grouped-expert prefill ...":
// top-k gate -> G128 quant -> permute -> gate_up GEMM -> SwiGLU requant -> down GEMM ->
// expert outputs stored in the output type -> combine -> output rounded to the output type
// (out_f32 != 0: float32, else bfloat16 values widened to float).  x [T, H] float (bf16
// values); out [T, H] float.  Returns 0.
int fo_moe_layer_forward(const float* logits, const float* x, int64_t T, int64_t H, int E,
                         int k, int64_t I, const uint8_t* w_gu, const float* s_gu,
                         const uint8_t* w_dn, const float* s_dn, int out_f32, float* out) {
  const int64_t R = T * k;
  std::vector<int32_t> ids(R), counts(E), offsets(E + 1), row_token(R), token_row(R);
  std::vector<float> gates(R), xs(T * (H / kGroup)), as(R * (H / kGroup));
  std::vector<uint8_t> xq(T * H), aq(R * H);
  fo_topk_gate(logits, T, E, k, ids.data(), gates.data());
  fo_quant_g128(x, T, H, xq.data(), xs.data());
  fo_moe_permute(ids.data(), T, k, E, xq.data(), xs.data(), H, counts.data(), offsets.data(),
                 row_token.data(), token_row.data(), aq.data(), as.data());
  std::vector<double> c(R * 2 * I);
  fo_grouped_gemm_w4a8(aq.data(), as.data(), offsets.data(), E, w_gu, s_gu, 2 * I, H, R, c.data());
  std::vector<uint8_t> hq(R * I);
  std::vector<float> hs(R * (I / kGroup)), h(R * I);
  fo_swiglu_requant(c.data(), R, I, hq.data(), hs.data(), h.data());
  c.clear();
  c.shrink_to_fit();
  std::vector<double> y(R * H);
  fo_grouped_gemm_w4a8(hq.data(), hs.data(), offsets.data(), E, w_dn, s_dn, H, I, R, y.data());
  std::vector<float> y_st(R * H);
  for (int64_t i = 0; i < R * H; ++i)
    y_st[i] = out_f32 ? static_cast<float>(y[i]) : bf16_to_float(bf16_bits(y[i]));
  std::vector<double> o(T * H);
  fo_moe_combine(y_st.data(), token_row.data(), gates.data(), T, k, H, o.data());
  for (int64_t i = 0; i < T * H; ++i)
    out[i] = out_f32 ? static_cast<float>(o[i]) : bf16_to_float(bf16_bits(o[i]));
  return 0;
}

// ---------------------------------------------------------------------- MXFP4 (E2M1)
// "[RFC] Support FP4 (E2M1) activation dispatch in MegaMoE": E2M1 activations for the
// dispatch buffer, consumed by an MXF4 main loop.  Readings (the page gives neither block nor
// scale format): the MX convention of blocks of 32 values along K with one power-of-two
// scale stored as E8M0 (code E + 127); E = floor(log2(amax)) - 2 (2 is the largest E2M1
// exponent), clamped at -127, which is also the code of an all-zero block; elements are the
// nearest E2M1 value of x / 2^E (ties to the even mantissa bit), saturating at 6, sign kept.
// Here the element code is found by a nearest-value search over the eight magnitudes.
void fo_mx_quant_e2m1(const float* x, int64_t M, int64_t K, uint8_t* packed, uint8_t* scales) {
  static const double mags[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  const int64_t nb = K / 32;
  for (int64_t r = 0; r < M; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* blk = x + r * K + b * 32;
      double amax = 0.0;
      for (int i = 0; i < 32; ++i) amax = std::fabs(static_cast<double>(blk[i])) > amax ? std::fabs(static_cast<double>(blk[i])) : amax;
      int E = -127;
      if (amax > 0.0) {
        int ex;
        std::frexp(amax, &ex);                 // amax = f * 2^ex, f in [0.5, 1)
        E = ex - 1 - 2;
        if (E < -127) E = -127;
      }
      scales[r * nb + b] = static_cast<uint8_t>(E + 127);
      for (int i = 0; i < 32; ++i) {
        const double v = std::ldexp(static_cast<double>(blk[i]), -E);
        const double a = std::fabs(v);
        int best = 7;
        if (a < 6.0) {
          best = 0;
          for (int c = 1; c < 8; ++c) {
            const double dc = std::fabs(a - mags[c]), db = std::fabs(a - mags[best]);
            if (dc < db || (dc == db && (c & 1) == 0)) best = c;
          }
        }
        const uint8_t code = static_cast<uint8_t>((std::signbit(v) ? 0x8 : 0x0) | best);
        const int64_t k = b * 32 + i;
        uint8_t& byte = packed[r * (K / 2) + (k >> 1)];
        if (k & 1) byte = static_cast<uint8_t>((byte & 0x0F) | (code << 4));
        else byte = static_cast<uint8_t>((byte & 0xF0) | code);
      }
    }
  }
}

// Grouped expert GEMM with MXFP4 activations: for expert e and its rows,
//   C[r, n] = sum_g sw[e, n, g] * sum_{k in g} a[r, k] * q[e, n, k],
//   a[r, k] = e2m1(code) * 2^(scale[r, k / 32] - 127).
// Here the E2M1 value is decoded from its fields (sign bit 3; exponent bits 2..1, bias 1;
// mantissa bit 0; exponent 0 is the subnormal step 0.5) and scaled with ldexp; plain loops,
// float64 throughout.  codes [R, K/2] (element 2b in the low nibble); scales [R, K/32].
static double e2m1_field_value(int code) {
  const int e = (code >> 1) & 3, m = code & 1;
  const double mag = e == 0 ? 0.5 * m : std::ldexp(1.0 + 0.5 * m, e - 1);
  return (code & 8) ? -mag : mag;
}

void fo_grouped_gemm_mxf4_w4(const uint8_t* codes, const uint8_t* scales, const int32_t* offsets,
                             int E, const uint8_t* w, const float* sw, int64_t N, int64_t K,
                             int64_t R, double* out) {
  const int64_t G = K / kGroup;
  for (int64_t i = 0; i < R * N; ++i) out[i] = 0.0;
  std::vector<double> arow(K);
  for (int e = 0; e < E; ++e) {
    const int64_t r0 = offsets[e], r1 = offsets[e + 1];
    for (int64_t r = r0; r < r1; ++r) {
      for (int64_t kk = 0; kk < K; ++kk) {
        const uint8_t byte = codes[r * (K / 2) + kk / 2];
        const int code = (kk & 1) ? (byte >> 4) : (byte & 0xF);
        arow[kk] = std::ldexp(e2m1_field_value(code), static_cast<int>(scales[r * (K / 32) + kk / 32]) - 127);
      }
      for (int64_t n = 0; n < N; ++n) {
        const uint8_t* wrow = w + (static_cast<int64_t>(e) * N + n) * (K / 2);
        double acc = 0.0;
        for (int64_t g = 0; g < G; ++g) {
          double part = 0.0;
          for (int64_t kk = g * kGroup; kk < (g + 1) * kGroup; ++kk) part += arow[kk] * int4_at(wrow, kk);
          acc += static_cast<double>(sw[(static_cast<int64_t>(e) * N + n) * G + g]) * part;
        }
        out[r * N + n] = acc;
      }
    }
  }
}

// ------------------------------------------------------------ stacked-layer helpers
// The stacked prefill workload's glue, not a page step.  Readings: a pre-norm block whose
// RMSNorm has unit gain and eps 1e-6, computed in float64 and rounded to bfloat16; router
// logits as float64 dot products rounded to float32; the attention core replaced by the
// identity on v with grouped-query sharing (query head h reads kv head h / (heads / kv_heads),
// head size 128).
void fo_rmsnorm(const float* h, int64_t T, int64_t H, float* out) {
  for (int64_t t = 0; t < T; ++t) {
    double ss = 0.0;
    for (int64_t c = 0; c < H; ++c) ss += static_cast<double>(h[t * H + c]) * h[t * H + c];
    const double inv = 1.0 / std::sqrt(ss / static_cast<double>(H) + 1e-6);
    for (int64_t c = 0; c < H; ++c)
      out[t * H + c] = bf16_to_float(bf16_bits(static_cast<double>(h[t * H + c]) * inv));
  }
}

void fo_router_logits(const float* xn, const float* w, int64_t T, int64_t H, int E, float* out) {
  for (int64_t t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int64_t c = 0; c < H; ++c) acc += static_cast<double>(xn[t * H + c]) * w[e * H + c];
      out[t * E + e] = static_cast<float>(acc);
    }
}

void fo_identity_attention(const float* v, int64_t T, int n_heads, int n_kv_heads, float* out) {
  const int rep = n_heads / n_kv_heads;
  for (int64_t t = 0; t < T; ++t)
    for (int h = 0; h < n_heads; ++h)
      for (int d = 0; d < 128; ++d)
        out[(t * n_heads + h) * 128 + d] = v[(t * n_kv_heads + h / rep) * 128 + d];
}

// Dense projection: dynamic activation quantization (per tensor, or one scale per row when
// rows != 0), the W8A8 GEMM, and the result rounded to bfloat16 ("feat(qwen4_exp) ...",
// sections "What this adds" and "Limits").  x [M, K]; wq [N, K]; out [M, N] float values.
void fo_linear_w8a8(const float* x, int64_t M, int64_t K, const uint8_t* wq, float sw,
                    int64_t N, int rows, float* out) {
  std::vector<uint8_t> q(M * K);
  std::vector<float> s(rows ? M : 1);
  if (rows) fo_quant_per_row(x, M, K, q.data(), s.data());
  else fo_quant_per_tensor(x, M, K, q.data(), s.data());
  std::vector<double> y(M * N);
  fo_linear_w8a8_gemm(q.data(), rows ? s.data() : nullptr, s[0], wq, sw, M, N, K, y.data());
  for (int64_t i = 0; i < M * N; ++i) out[i] = bf16_to_float(bf16_bits(y[i]));
}

// The per-token int4 expert dispatch that the grouped GEMM replaces ("FP8 grouped-expert
// prefill ...", section 1: one dispatch per routed token per layer).  Reading: activations
// stay unquantized; for each routed (token, slot) the expert FFN y = Wd (silu(Wg x) * (Wu x))
// runs with the int4 weights dequantized as q * scale, in float64, token by token; the
// output is the gate-weighted sum in slot order, rounded to the output type.
void fo_moe_layer_int4_baseline(const float* logits, const float* x, int64_t T, int64_t H, int E,
                                int k, int64_t I, const uint8_t* w_gu, const float* s_gu,
                                const uint8_t* w_dn, const float* s_dn, int out_f32, float* out) {
  std::vector<int32_t> ids(T * k);
  std::vector<float> gates(T * k);
  fo_topk_gate(logits, T, E, k, ids.data(), gates.data());
  const int64_t Gh = H / kGroup, Gi = I / kGroup;
  std::vector<double> c(2 * I), hmid(I), acc(H);
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t o = 0; o < H; ++o) acc[o] = 0.0;
    for (int j = 0; j < k; ++j) {
      const int e = ids[t * k + j];
      for (int64_t n = 0; n < 2 * I; ++n) {
        const uint8_t* wrow = w_gu + (static_cast<int64_t>(e) * 2 * I + n) * (H / 2);
        const float* srow = s_gu + (static_cast<int64_t>(e) * 2 * I + n) * Gh;
        double d = 0.0;
        for (int64_t kk = 0; kk < H; ++kk)
          d += static_cast<double>(x[t * H + kk]) * (int4_at(wrow, kk) * static_cast<double>(srow[kk / kGroup]));
        c[n] = d;
      }
      for (int64_t i = 0; i < I; ++i) hmid[i] = c[i] / (1.0 + std::exp(-c[i])) * c[I + i];
      for (int64_t o = 0; o < H; ++o) {
        const uint8_t* wrow = w_dn + (static_cast<int64_t>(e) * H + o) * (I / 2);
        const float* srow = s_dn + (static_cast<int64_t>(e) * H + o) * Gi;
        double d = 0.0;
        for (int64_t i = 0; i < I; ++i)
          d += hmid[i] * (int4_at(wrow, i) * static_cast<double>(srow[i / kGroup]));
        acc[o] += static_cast<double>(gates[t * k + j]) * d;
      }
    }
    for (int64_t o = 0; o < H; ++o)
      out[t * H + o] = out_f32 ? static_cast<float>(acc[o]) : bf16_to_float(bf16_bits(acc[o]));
  }
}

}  // extern "C"
