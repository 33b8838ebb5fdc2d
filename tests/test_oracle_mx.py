"""Pins of the MXFP4 (E2M1 + per-32 power-of-two scale) oracle against closed forms and
brute force (no GPU)."""

import numpy as np
import pytest

from oracle.mx import (E2M1_MAX, MX_BLOCK, e2m1_decode, e2m1_encode, mx_block_exponent,
                       mx_dequant_e2m1, mx_quant_e2m1)

# E2M1 values by code: 1 sign, 2 exponent (bias 1), 1 mantissa bit; written out by hand
E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
               -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def _nearest_even(v):
    """Brute force: the E2M1 code nearest to v; on a tie the one with mantissa bit 0;
    beyond 6 the largest magnitude."""
    sign = 0x8 if np.signbit(v) else 0x0
    a = abs(v)
    if a > E2M1_MAX:
        return sign | 0x7
    dists = [abs(a - abs(E2M1_VALUES[c])) for c in range(8)]
    best = min(dists)
    cands = [c for c in range(8) if dists[c] == best]
    if len(cands) > 1:
        cands = [c for c in cands if c % 2 == 0]
    return sign | cands[0]


def test_decode_table():
    for c in range(16):
        v = e2m1_decode(c)
        assert v == E2M1_VALUES[c] and np.signbit(v) == np.signbit(E2M1_VALUES[c])


def test_roundtrip_every_code():
    for c in range(16):
        assert e2m1_encode(e2m1_decode(c)) == c


def test_encode_ties_and_saturation():
    # midpoints between neighbours go to the even mantissa
    assert e2m1_encode(0.25) == 0x0 and e2m1_encode(0.75) == 0x2
    assert e2m1_encode(1.25) == 0x2 and e2m1_encode(1.75) == 0x4
    assert e2m1_encode(2.5) == 0x4 and e2m1_encode(3.5) == 0x6
    assert e2m1_encode(5.0) == 0x6
    assert e2m1_encode(-5.0) == 0xE
    # beyond the largest magnitude: saturate
    for v in (6.01, 7.99, 8.0, 1e30):
        assert e2m1_encode(v) == 0x7 and e2m1_encode(-v) == 0xF
    # zero keeps its sign
    assert e2m1_encode(0.0) == 0x0 and e2m1_encode(-0.0) == 0x8 and e2m1_encode(-0.1) == 0x8


def test_encode_matches_brute_force():
    rng = np.random.default_rng(3)
    grid = np.arange(-8 * 64, 8 * 64 + 1) / 64.0          # every multiple of 1/64 in [-8, 8]
    vals = np.concatenate([grid, rng.uniform(-9, 9, 4000), rng.uniform(-1, 1, 2000)])
    for v in vals:
        assert e2m1_encode(v) == _nearest_even(v), v


def test_block_exponent_closed_form():
    assert mx_block_exponent(6.0) == 0
    assert mx_block_exponent(4.0) == 0
    assert mx_block_exponent(7.99) == 0
    assert mx_block_exponent(8.0) == 1
    assert mx_block_exponent(3.99) == -1
    assert mx_block_exponent(1.0) == -2
    assert mx_block_exponent(2.0 ** -100) == -102
    assert mx_block_exponent(2.0 ** -130) == -127      # clamped: scale code 0
    assert mx_block_exponent(0.0) == -127
    # the block's largest magnitude lands in [4, 8) before the cast
    rng = np.random.default_rng(5)
    for a in rng.uniform(1e-6, 1e6, 500):
        e = mx_block_exponent(a)
        assert 4.0 <= a / 2.0 ** e < 8.0


def test_quant_representable_block_is_exact():
    # a block of E2M1 values times 2^E with its largest magnitude 6 * 2^E round-trips
    rng = np.random.default_rng(7)
    for e in (-20, -3, 0, 5):
        codes = rng.integers(0, 16, size=(2, MX_BLOCK))
        vals = np.array([[e2m1_decode(c) for c in row] for row in codes]) * 2.0 ** e
        vals[:, 0] = 6.0 * 2.0 ** e
        packed, scales = mx_quant_e2m1(vals)
        assert np.all(scales == e + 127)
        np.testing.assert_array_equal(mx_dequant_e2m1(packed, scales), vals)


def test_quant_packing_order_and_zero_block():
    x = np.zeros((1, 64))
    x[0, 0] = 1.0      # block 0: amax 1 -> E = -2, element 0 -> 4 (code 6)
    x[0, 1] = -0.5     # -> -2 (code 0xC)
    packed, scales = mx_quant_e2m1(x)
    assert packed[0, 0] == 0x6 | (0xC << 4)
    assert scales[0, 0] == 125 and scales[0, 1] == 0    # block 1 is all zero
    assert np.all(packed[0, 16:] == 0)


def test_quant_error_bound():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((4, 256)) * np.exp(rng.uniform(-8, 8, size=(4, 1)))
    x[1, 5] = 1e4                                          # an outlier in one block
    packed, scales = mx_quant_e2m1(x)
    dq = mx_dequant_e2m1(packed, scales)
    xs = 2.0 ** (np.repeat(scales.astype(np.float64), MX_BLOCK, axis=1) - 127.0)
    a = np.abs(x) / xs                                     # scaled magnitude, < 8
    half_step = np.where(a < 2.0, 0.25, np.where(a < 4.0, 0.5, 1.0))
    err = np.abs(dq - x) / xs
    sat = a > E2M1_MAX
    assert np.all(err[~sat] <= half_step[~sat])
    assert np.all(np.abs(dq[sat]) == E2M1_MAX * xs[sat])
    assert np.all(a < 8.0)


@pytest.mark.parametrize("seed", [0, 1])
def test_quant_matches_per_element_definition(seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((3, 96)).astype(np.float32).astype(np.float64)
    packed, scales = mx_quant_e2m1(x)
    for i in range(3):
        for j in range(96):
            b = j // MX_BLOCK
            e = mx_block_exponent(np.max(np.abs(x[i, b * MX_BLOCK:(b + 1) * MX_BLOCK])))
            code = (packed[i, j // 2] >> (4 * (j % 2))) & 0xF
            assert code == _nearest_even(x[i, j] / 2.0 ** e)
