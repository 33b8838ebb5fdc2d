"""Oracle: E2M1 (FP4) activations with a power-of-two scale per 32 values (MXFP4).

Test infrastructure only (see the package docstring).  float64 throughout; every value
the method produces here is exact in float64, so no rounding order is involved.

Source: "[RFC] Support FP4 (E2M1) activation dispatch in MegaMoE" proposes E2M1 activations
for the expert dispatch buffer (half the bytes of e4m3) and names the MXF4 main loop as the
consumer.  The page gives neither the block size nor the scale format.  Reading: the MX
convention that "MXF4" refers to -- blocks of 32 consecutive values along K, one shared
scale per block stored as an 8-bit biased power of two (E8M0), elements in E2M1 -- and the
usual choice of that shared exponent: floor(log2(amax)) minus the largest E2M1 exponent (2),
so that the block's largest magnitude lands in [4, 8) before the cast.  Further readings:
round to nearest, ties to even; magnitudes above 6 saturate to 6; a zero result keeps the
sign of its input; the exponent is clamped at -127 (scale code 0), which is also the code of
an all-zero block.
"""

import numpy as np

from .fp8 import int4_unpack

E2M1_MAX = 6.0
MX_BLOCK = 32
# the eight E2M1 magnitudes, indexed by the 3-bit code (exponent bits 2..1, mantissa bit 0)
_MAGS = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def e2m1_decode(code):
    """Value of a 4-bit E2M1 code: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0;
    exponent field 0 is the subnormal range (m * 0.5)."""
    code = int(code) & 0xF
    sign = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return sign * 0.5 * m
    return sign * (1.0 + 0.5 * m) * 2.0 ** (e - 1)


def e2m1_encode(v):
    """E2M1 code of a float64 value: round to nearest, ties to the code with an even
    mantissa bit, saturating at 6.  Works on the exponent/mantissa split, not on a table
    search."""
    v = float(v)
    sign = 0x8 if np.signbit(v) else 0x0
    a = abs(v)
    if a >= E2M1_MAX:
        return sign | 0x7
    if a < 1.0:
        # subnormal step 0.5: q = a / 0.5 in [0, 2), round half to even
        q = a * 2.0
        n = np.floor(q)
        r = q - n
        if r > 0.5 or (r == 0.5 and int(n) % 2 == 1):
            n += 1
        n = int(n)
        if n == 2:  # rounded up into the normal range: 1.0
            return sign | 0x2
        return sign | n
    # normal: a = (1 + f) * 2^e with e in {0, 1, 2}; one mantissa bit -> step 2^(e - 1)
    e = int(np.floor(np.log2(a)))
    e = min(e, 2)
    step = 2.0 ** (e - 1)
    q = a / step              # in [2, 4): mantissa 2 + m with m in {0, 1}, plus a fraction
    n = np.floor(q)
    r = q - n
    if r > 0.5 or (r == 0.5 and int(n) % 2 == 1):
        n += 1
    n = int(n)
    if n == 4:                # carried into the next binade
        e += 1
        n = 2
    if e > 2:
        return sign | 0x7
    return sign | ((e + 1) << 1) | (n - 2)


def mx_block_exponent(amax):
    """Shared exponent E of a block: floor(log2(amax)) - 2, clamped at -127 (and -127 for an
    all-zero block).  The stored scale code is E + 127."""
    amax = float(amax)
    if amax == 0.0:
        return -127
    m, e = np.frexp(amax)     # amax = m * 2^e, m in [0.5, 1): floor(log2(amax)) = e - 1
    return max(int(e) - 1 - 2, -127)


def mx_quant_e2m1(x):
    """MXFP4 quantization of activations x [M, K] (float64 values of bf16 inputs, K % 32 == 0).

    Returns (codes uint8 [M, K/2], scales uint8 [M, K/32]): byte b of a row holds elements
    2b (low nibble) and 2b + 1 (high nibble); scale code c means 2^(c - 127).  Each element
    is e2m1_encode(x / 2^E) with E the block's mx_block_exponent.
    """
    x = np.asarray(x, dtype=np.float64)
    m, k = x.shape
    assert k % MX_BLOCK == 0
    codes = np.zeros((m, k), dtype=np.uint8)
    scales = np.zeros((m, k // MX_BLOCK), dtype=np.uint8)
    for i in range(m):
        for b in range(k // MX_BLOCK):
            blk = x[i, b * MX_BLOCK:(b + 1) * MX_BLOCK]
            e = mx_block_exponent(np.max(np.abs(blk)))
            scales[i, b] = e + 127
            inv = 2.0 ** (-e)
            for j in range(MX_BLOCK):
                codes[i, b * MX_BLOCK + j] = e2m1_encode(blk[j] * inv)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, scales


def mx_dequant_e2m1(packed, scales):
    """Values of MXFP4 activations: decode(code) * 2^(scale - 127), float64 [M, K]."""
    packed = np.asarray(packed, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    m, kh = packed.shape
    k = kh * 2
    out = np.empty((m, k), dtype=np.float64)
    table = np.array([e2m1_decode(c) for c in range(16)])
    out[:, 0::2] = table[packed & 0xF]
    out[:, 1::2] = table[packed >> 4]
    sc = 2.0 ** (scales.astype(np.float64) - 127.0)
    return out * np.repeat(sc, MX_BLOCK, axis=1)


def grouped_gemm_mxf4_w4(codes, scales, offsets, w_packed, w_scale):
    """Grouped expert GEMM with MXFP4 activations and the int4 expert banks.

    "[RFC] Support FP4 (E2M1) activation dispatch in MegaMoE": the dispatched activations are
    E2M1 with a shared scale per block and the expert GEMM consumes them in its MX main loop
    (there, mxf8f6f4 with K = 32 per step when the other operand is 8-bit).  Reading: the
    weight side stays this method's int4 bank with its per-(output row, 128-K group) scale,
    which is applied to each group's partial sum as in grouped_gemm_w4a8; the activation
    side carries one power-of-two scale per 32 values inside the group.  Definition written
    out: for expert e and its rows r in [offsets[e], offsets[e+1]),
        C[r, n] = sum_g  sw[e, n, g] * sum_{k in group g} a[r, k] * q[e, n, k],
        a[r, k] = dec(code[r, k]) * 2^(scale[r, k // 32] - 127).
    Products have at most 5 significant bits, so each group sum is exact in float64 unless
    the four block scales of a group span more than about 45 binades; the weight scaling and
    the outer sum are float64.

    codes uint8 [R, K/2] (element 2b in the low nibble of byte b); scales uint8 [R, K/32];
    offsets int [E+1]; w_packed uint8 [E, N, K/2]; w_scale float32 [E, N, K/128].
    Returns float64 [R, N] (rows past offsets[E] are zero).
    """
    a = mx_dequant_e2m1(codes, scales)
    r_total, kdim = a.shape
    e_count, n, _ = np.asarray(w_packed).shape
    groups = kdim // 128
    out = np.zeros((r_total, n), dtype=np.float64)
    for e in range(e_count):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            continue
        w = int4_unpack(w_packed[e], kdim).astype(np.float64)
        sw = np.asarray(w_scale[e], dtype=np.float64)
        for g in range(groups):
            ks = slice(g * 128, (g + 1) * 128)
            out[r0:r1] += (a[r0:r1, ks] @ w[:, ks].T) * sw[None, :, g]
    return out
