"""Oracle: e4m3 codec, int4 nibble format, bf16 rounding and activation quantization.

Test infrastructure only (see the package docstring).  float64 throughout, except where a
step is defined in float32 (the scale and the division x/s), where numpy float32 IEEE
arithmetic is used on purpose.
"""

import numpy as np

E4M3_MAX = 448.0          # largest finite e4m3 (E4M3FN) magnitude: code 0x7E = 1.75 * 2^8
F32_MIN_NORMAL = np.float32(2.0 ** -126)


def e4m3_decode_table():
    """Value of each of the 256 e4m3 codes, as float64 (NaN for the two NaN codes).

    Format: 1 sign bit, 4 exponent bits, 3 mantissa bits ("FP8 vs INT4 KV Cache: How to
    Achieve Sub-10ms MoE Serving", section "FP8 (E4M3) vs. Grouped INT4", item 1).  The
    pages do not give the bias or the special codes; reading: the OCP E4M3FN variant that
    FP8 tensor cores implement -- bias 7, subnormals at exponent field 0, no infinities,
    S.1111.111 is NaN, so the largest finite value is 448 (the divisor of the amax/448
    scale on the "Module fp8_ffi" page).
    """
    vals = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        exp_field = (code >> 3) & 0xF
        mant = code & 0x7
        if exp_field == 0xF and mant == 0x7:
            vals[code] = np.nan
        elif exp_field == 0:
            vals[code] = sign * (mant / 8.0) * 2.0 ** -6
        else:
            vals[code] = sign * (1.0 + mant / 8.0) * 2.0 ** (exp_field - 7)
    return vals


_TABLE = e4m3_decode_table()
_POS_VALUES = _TABLE[0:0x7F].copy()     # codes 0x00..0x7E: 0 .. 448, strictly increasing


def e4m3_decode(codes):
    """uint8 codes -> float64 values (table lookup)."""
    return _TABLE[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(x):
    """float32 values -> e4m3 codes (uint8), round to nearest even, saturating.

    Rounding is on the exact float32 value: the quantum of the binade [2^E, 2^(E+1)) is
    2^(E-3) (3 mantissa bits), and 2^-9 below 2^-6 (subnormals).  Magnitudes that round
    above 448 become 448 (saturating cast, matching the "satfinite" conversion that the
    e4m3 tensor-core path provides).  The sign is kept, so -0.0 encodes as 0x80.  Inputs are
    assumed finite; +-inf saturate like large values.  NaN inputs are not defined here.
    """
    x64 = np.asarray(x, dtype=np.float32).astype(np.float64)
    neg = np.signbit(x64)
    a = np.abs(x64)
    a = np.where(np.isinf(a), 2.0 * E4M3_MAX, a)
    _, e = np.frexp(a)                 # a = m * 2^e with m in [0.5, 1)
    binade = np.maximum(e - 1, -6)     # a in [2^binade, 2^(binade+1)); subnormal floor -6
    quantum = np.ldexp(1.0, binade - 3)
    q = np.rint(a / quantum) * quantum  # a/quantum is exact (power-of-two quantum); rint = RNE
    q = np.minimum(q, E4M3_MAX)
    mag_code = np.searchsorted(_POS_VALUES, q)
    if not np.array_equal(_POS_VALUES[np.minimum(mag_code, 0x7E)], q):
        raise AssertionError("e4m3_encode produced a value that is not an e4m3 magnitude")
    return (mag_code.astype(np.uint8) | (neg.astype(np.uint8) << 7)).astype(np.uint8)


def int4_unpack(packed, k):
    """Packed int4 bank -> int8 values in -8..7, shape [..., k].

    Format ("FP8 grouped-expert prefill with on-chip int4-to-e4m3 dequant", section 1: a
    resident packed-int4 weight bank, two values per byte).  Readings, the pages being
    silent: values are two's complement nibbles; byte b of a row holds element 2b in its low
    nibble and element 2b+1 in its high nibble (low nibble first, the extraction order of
    the unpack routine on the "FP8 vs INT4 KV Cache" page).
    """
    p = np.asarray(packed, dtype=np.uint8)
    lo = (p & 0x0F).astype(np.int16)
    hi = (p >> 4).astype(np.int16)
    lo = np.where(lo >= 8, lo - 16, lo)
    hi = np.where(hi >= 8, hi - 16, hi)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.int8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    if out.shape[-1] != k:
        raise ValueError("packed row length does not match k")
    return out


def bf16_round(x):
    """float64 -> nearest bfloat16 (ties to even), returned as uint16 bit patterns.

    bfloat16 keeps 8 significant bits; the quantum of binade [2^E, 2^(E+1)) is 2^(E-7), and
    2^-133 below 2^-126.  Finite inputs only (the outputs here never approach 2^128).
    """
    x64 = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x64)
    a = np.abs(x64)
    _, e = np.frexp(a)
    binade = np.maximum(e - 1, -126)
    quantum = np.ldexp(1.0, binade - 7)
    q = np.rint(a / quantum) * quantum
    q32 = q.astype(np.float32)              # exact: q has <= 8 significant bits
    if not np.array_equal(q32.astype(np.float64), q):
        raise AssertionError("bf16_round: value not representable in float32")
    bits = (q32.view(np.uint32) >> 16).astype(np.uint16)
    return bits | (neg.astype(np.uint16) << 15)


def bf16_bits_to_f32(bits):
    """uint16 bfloat16 bit patterns -> float32 values (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def _scale_from_amax(amax):
    """Per-group (or per-tensor) scale s = amax / 448 in float32, with the zero floor.

    "Module fp8_ffi" (module doc): one scalar scale amax/448 per batch; "feat(qwen4_exp):
    load-time per-tensor FP8 dense projections", section "Testing": the op has a zero-input
    scale floor, whose value the page does not print.  Readings: the division is the IEEE
    float32 one; amax == 0 gives s = 1 (every code is then 0x00); a scale below the smallest
    normal float32 (2^-126) is raised to 2^-126.
    """
    amax = np.asarray(amax, dtype=np.float32)
    s = amax / np.float32(E4M3_MAX)
    s = np.where(amax == 0, np.float32(1.0), s)
    s = np.where(s < F32_MIN_NORMAL, F32_MIN_NORMAL, s)
    return s.astype(np.float32)


def quant_act_g128(x_f32):
    """Activation quantization per (token, 128-element K group).

    "FP8 grouped-expert prefill with on-chip int4-to-e4m3 dequant", section 1: activations
    quantized to e4m3 with a per-(token, group) scale.  Steps: amax = max|x| over the 128
    values of the group; s = fp32(amax / 448); q = e4m3_rne_sat(fp32(x / s)).
    Reading: the code is taken from the float32 quotient x / s (IEEE division, then the
    e4m3 rounding) rather than from x times a reciprocal -- x / s is the definition.

    x_f32: [M, K] float32 (bf16 inputs widened exactly), K a multiple of 128.
    Returns (codes uint8 [M, K], scales float32 [M, K/128]).
    """
    x = np.asarray(x_f32, dtype=np.float32)
    m, k = x.shape
    if k % 128:
        raise ValueError("K must be a multiple of 128")
    g = x.reshape(m, k // 128, 128)
    amax = np.max(np.abs(g), axis=2)
    s = _scale_from_amax(amax)
    q = e4m3_encode(g / s[:, :, None])
    return q.reshape(m, k), s


def quant_act_per_tensor(x_f32):
    """Dynamic per-tensor activation quantization: one amax over the whole [M, K] tensor.

    "feat(qwen4_exp): load-time per-tensor FP8 dense projections", section "What this adds"
    (amax pass, then the cast, no host sync) and "Module fp8_ffi" (amax reduce, scale
    finalize, e4m3 quantize).  Same scale rule and rounding as ``quant_act_g128``.
    Returns (codes uint8 [M, K], scale float32 scalar).
    """
    x = np.asarray(x_f32, dtype=np.float32)
    amax = np.max(np.abs(x)) if x.size else np.float32(0.0)
    s = _scale_from_amax(amax)
    q = e4m3_encode(x / s)
    return q, np.float32(s)


def quant_act_per_row(x_f32):
    """Dynamic activation quantization with one scale per row (token).

    "feat(qwen4_exp): load-time per-tensor FP8 dense projections", section "Limits": the
    row-wise alternative to one per-tensor scale, so that an outlier channel in one row no
    longer sets the scale of every row.  Same scale rule and rounding as
    ``quant_act_per_tensor``, with the amax taken over each row's K values.
    Returns (codes uint8 [M, K], scales float32 [M]).
    """
    x = np.asarray(x_f32, dtype=np.float32)
    m, k = x.shape
    amax = np.max(np.abs(x), axis=1) if k else np.zeros(m, dtype=np.float32)
    s = _scale_from_amax(amax)
    q = e4m3_encode(x / s[:, None])
    return q, s
