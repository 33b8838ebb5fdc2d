"""Pins for the oracle's e4m3 codec, int4 format, bf16 rounding and activation quant.

Each expected value below comes from the e4m3 / bf16 format definitions worked by hand (the
derivation is in the comment beside it), from a library conversion (torch's CPU float8 and
bfloat16 casts), or from an invariant -- never from the oracle itself.
"""

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8 as ofp8
from workloads import pack_int4

# --- e4m3 decode table -------------------------------------------------------------------

@pytest.mark.parametrize("code,value", [
    (0x00, 0.0),
    (0x01, 2.0 ** -9),            # smallest subnormal: 1/8 * 2^-6
    (0x07, 7 * 2.0 ** -9),        # largest subnormal
    (0x08, 2.0 ** -6),            # smallest normal
    (0x38, 1.0),                  # exponent field 7 = bias
    (0x3F, 1.875),                # 1 + 7/8
    (0x40, 2.0),
    (0x7E, 448.0),                # 1.75 * 2^8, largest finite
    (0xB8, -1.0),
    (0xFE, -448.0),
])
def test_decode_closed_form_points(code, value):
    assert oracle.e4m3_decode(np.uint8(code)) == value


def test_decode_special_codes():
    t = oracle.e4m3_decode_table()
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert t[0x80] == 0.0 and np.signbit(t[0x80])
    assert np.sum(np.isfinite(t)) == 254


def test_decode_table_structure():
    t = oracle.e4m3_decode_table()
    pos = t[0:0x7F]
    assert np.all(np.diff(pos) > 0)                      # strictly increasing magnitudes
    assert np.array_equal(t[0x80:0xFF], -pos)            # sign bit negates
    # inside exponent field e >= 1 the spacing is 2^(e-10); subnormal spacing 2^-9
    for e in range(1, 16):
        codes = [(e << 3) | m for m in range(8) if (e << 3) | m < 0x7F]
        steps = np.diff(t[codes])
        assert np.all(steps == 2.0 ** (e - 10))
    assert np.all(np.diff(t[0:9]) == 2.0 ** -9)


# --- e4m3 encode -------------------------------------------------------------------------

def test_encode_roundtrips_every_finite_code():
    t = oracle.e4m3_decode_table()
    codes = np.array([c for c in range(256) if np.isfinite(t[c])], dtype=np.uint8)
    vals = t[codes].astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def test_encode_matches_torch_cast_in_range():
    # torch's CPU float8_e4m3fn cast rounds to nearest even; it does not saturate, so the
    # comparison stays inside +-464 (the rounding boundary above 448).
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.uniform(-464, 464, 200_000),
        rng.standard_normal(200_000) * 3,
        rng.standard_normal(100_000) * 2.0 ** -8,
        np.ldexp(rng.uniform(-1, 1, 100_000), rng.integers(-12, 9, 100_000)),
    ]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x), ref)


def test_encode_ties_go_to_even_code():
    t = oracle.e4m3_decode_table()
    pos = t[0:0x7F]
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)    # exact in float32
    assert np.array_equal(mids.astype(np.float64), (pos[:-1] + pos[1:]) / 2)
    got = oracle.e4m3_encode(mids)
    lower = np.arange(0, 0x7E, dtype=np.uint8)
    expect = np.where(lower % 2 == 0, lower, lower + 1).astype(np.uint8)
    assert np.array_equal(got, expect)


def test_encode_saturates_and_keeps_sign():
    big = np.array([448, 449, 463.9, 464, 465, 480, 1e6, 3e38, np.inf], dtype=np.float32)
    assert np.all(oracle.e4m3_encode(big) == 0x7E)
    assert np.all(oracle.e4m3_encode(-big) == 0xFE)
    assert oracle.e4m3_encode(np.float32(-0.0)) == 0x80
    # below half the smallest subnormal -> signed zero; exactly half -> ties to even (0)
    assert oracle.e4m3_encode(np.float32(2.0 ** -10)) == 0x00
    assert oracle.e4m3_encode(np.float32(-(2.0 ** -10))) == 0x80
    # 0.75 of the smallest subnormal rounds up to it
    assert oracle.e4m3_encode(np.float32(3 * 2.0 ** -11)) == 0x01


def test_encode_subnormal_rounding():
    # 1.5 * 2^-9 is a tie between codes 0x01 (odd) and 0x02 (even) -> 0x02
    assert oracle.e4m3_encode(np.float32(1.5 * 2.0 ** -9)) == 0x02
    # 2.5 * 2^-9 is a tie between 0x02 (even) and 0x03 -> 0x02
    assert oracle.e4m3_encode(np.float32(2.5 * 2.0 ** -9)) == 0x02
    # 7.5 * 2^-9 is a tie between 0x07 and 0x08 (= 2^-6, even) -> 0x08
    assert oracle.e4m3_encode(np.float32(7.5 * 2.0 ** -9)) == 0x08


# --- int4 in e4m3 ------------------------------------------------------------------------

def test_int4_values_are_exact_e4m3_codes():
    # hand-derived codes (bias 7): 1 = 1.0*2^0 -> 0 0111 000; 3 = 1.5*2^1 -> 0 1000 100;
    # 5 = 1.25*2^2 -> 0 1001 010; 7 = 1.75*2^2 -> 0 1001 110; 8 = 1.0*2^3 -> 0 1010 000
    expect = {0: 0x00, 1: 0x38, 2: 0x40, 3: 0x44, 4: 0x48, 5: 0x4A, 6: 0x4C, 7: 0x4E,
              -1: 0xB8, -2: 0xC0, -3: 0xC4, -4: 0xC8, -5: 0xCA, -6: 0xCC, -7: 0xCE, -8: 0xD0}
    for q, code in expect.items():
        assert oracle.e4m3_encode(np.float32(q)) == code
        assert oracle.e4m3_decode(np.uint8(code)) == q


def test_int4_nibble_order_and_sign():
    packed = np.array([[0x21, 0x8F, 0x7F]], dtype=np.uint8)
    # 0x21: low nibble 1 (k=0), high nibble 2 (k=1); 0x8F: low 0xF = -1, high 0x8 = -8
    assert oracle.int4_unpack(packed, 6).tolist() == [[1, 2, -1, -8, -1, 7]]
    rng = np.random.default_rng(2)
    q = rng.integers(-8, 8, size=(3, 5, 256))
    assert np.array_equal(oracle.int4_unpack(pack_int4(q), 256), q)


# --- bf16 rounding -----------------------------------------------------------------------

def test_bf16_round_matches_torch_from_float32():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(100_000) * 10,
                        np.ldexp(rng.uniform(-1, 1, 50_000), rng.integers(-130, 60, 50_000))]
                       ).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.bf16_round(x.astype(np.float64)), ref)


def test_bf16_round_single_rounding_from_float64():
    # 1 + 2^-8 + 2^-30 lies above the midpoint 1 + 2^-8, so the nearest bf16 is 1 + 2^-7
    # (bits 0x3F81); rounding through float32 first would land on the tie and give 1.0.
    assert oracle.bf16_round(np.float64(1 + 2.0 ** -8 + 2.0 ** -30)) == 0x3F81
    assert oracle.bf16_round(np.float64(1 + 2.0 ** -8)) == 0x3F80
    assert oracle.bf16_round(np.float64(-2.0)) == 0xC000


# --- activation quantization --------------------------------------------------------------

def test_quant_zero_group_gives_zero_codes_and_unit_scale():
    q, s = oracle.quant_act_g128(np.zeros((3, 256), np.float32))
    assert np.all(q == 0) and np.all(s == 1.0)
    q, s = oracle.quant_act_per_tensor(np.zeros((3, 256), np.float32))
    assert np.all(q == 0) and s == 1.0


def test_quant_closed_form_group():
    # x_i = (7/64) * i, i = 1..128: amax = 14, s = 14/448 = 1/32 exactly, x/s = 3.5 i.
    x = (np.arange(1, 129, dtype=np.float32) * np.float32(7 / 64))[None, :]
    q, s = oracle.quant_act_g128(x)
    assert s[0, 0] == np.float32(1 / 32)
    # 3.5 = 1.75*2 -> 0 1000 110 = 0x46;  7 -> 0x4E;  10.5: tie between 10 (m=2) and 11
    # (m=3) in [8,16) -> 10 = 0 1010 010 = 0x52;  17.5: quantum 2 -> 18 = 1.125*16 ->
    # 0 1011 001 = 0x59;  24.5 -> 24 = 1.5*16 -> 0x5C;  448 -> 0x7E
    for i, code in [(1, 0x46), (2, 0x4E), (3, 0x52), (5, 0x59), (7, 0x5C), (128, 0x7E)]:
        assert q[0, i - 1] == code, i
    qn, sn = oracle.quant_act_g128(-x)
    assert np.array_equal(qn, q | 0x80) and sn[0, 0] == s[0, 0]


def test_quant_tiny_group_scale_floor():
    x = np.zeros((1, 128), np.float32)
    x[0, 5] = np.float32(1e-40)                     # a float32 subnormal
    q, s = oracle.quant_act_g128(x)
    assert s[0, 0] == np.float32(2.0 ** -126)
    assert abs(oracle.e4m3_decode(q[0, 5]) * float(s[0, 0]) - 1e-40) < 2.0 ** -126 * 2.0 ** -9


def test_per_tensor_equals_group_mode_on_one_group():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((1, 128)).astype(np.float32)
    qg, sg = oracle.quant_act_g128(x)
    qt, st = oracle.quant_act_per_tensor(x)
    assert np.array_equal(qg, qt) and sg[0, 0] == st


def test_quant_error_bound():
    # RNE into 3 mantissa bits: relative error <= 2^-4 for |x/s| >= 2^-6, absolute error
    # <= s * 2^-10 below that.  The amax element lands exactly on +-448.
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((64, 512)) * np.exp(rng.uniform(-6, 6, (64, 1)))).astype(np.float32)
    q, s = oracle.quant_act_g128(x)
    srep = np.repeat(s, 128, axis=1).astype(np.float64)
    deq = oracle.e4m3_decode(q) * srep
    err = np.abs(deq - x.astype(np.float64))
    bound = np.maximum(np.abs(x) * 2.0 ** -4, srep * 2.0 ** -10) * (1 + 1e-6)
    assert np.all(err <= bound)
    g = np.abs(x.reshape(64, 4, 128))
    top = np.argmax(g, axis=2)
    qg = q.reshape(64, 4, 128)
    assert np.all(np.take_along_axis(qg, top[..., None], 2) & 0x7F == 0x7E)


# --- per-row (row-wise) activation quant ---------------------------------------------------

def test_per_row_equals_per_tensor_on_each_row():
    # a row is a tensor of its own: the per-row mode must give, row by row, what the
    # independent per-tensor function gives for that row alone
    rng = np.random.default_rng(21)
    x = (rng.standard_normal((6, 384)) * np.exp(rng.uniform(-5, 5, (6, 1)))).astype(np.float32)
    q, s = oracle.quant_act_per_row(x)
    assert q.shape == x.shape and s.shape == (6,)
    for i in range(6):
        qt, st = oracle.quant_act_per_tensor(x[i:i + 1])
        assert np.array_equal(q[i:i + 1], qt) and s[i] == st


def test_per_row_equals_group_mode_when_k_is_128():
    rng = np.random.default_rng(22)
    x = rng.standard_normal((9, 128)).astype(np.float32)
    qr, sr = oracle.quant_act_per_row(x)
    qg, sg = oracle.quant_act_g128(x)
    assert np.array_equal(qr, qg) and np.array_equal(sr, sg[:, 0])


def test_per_row_zero_row_and_amax_code():
    x = np.zeros((3, 256), dtype=np.float32)
    x[1, 7] = -3.0                       # amax 3 -> s = 3/448; x/s = -448 -> code 0xFE
    x[2] = np.linspace(-1.0, 2.0, 256, dtype=np.float32)  # amax 2 at the last element -> 0x7E
    q, s = oracle.quant_act_per_row(x)
    assert np.all(q[0] == 0) and s[0] == np.float32(1.0)
    assert s[1] == np.float32(3.0) / np.float32(448.0) and q[1, 7] == 0xFE
    assert np.count_nonzero(q[1]) == 1
    assert q[2, 255] == 0x7E
