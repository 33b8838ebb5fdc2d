"""Pins of the oracle's grouped GEMM with MXFP4 activations (oracle.grouped_gemm_mxf4_w4).

1. Closed form: with every activation code 1.0 and one non-zero int4 weight per output
   column, each output is the weight's group scale times 2^(the activation scale of the
   32-value block that holds that weight's k, minus 127).  A wrong block index (k // 16,
   k // 128), a wrong bias or a wrong weight group fails it.
2. Equivalence with the W4A8 grouped GEMM, itself pinned by exact and closed-form cases:
   when the four block scales of each 128-group are equal, an MXFP4 row is an e4m3 row
   (every E2M1 value is exact in e4m3) with that power of two as its G128 scale.
3. Routing structure: rows past offsets[E] stay zero, an expert with no rows contributes
   nothing, and each expert's rows use that expert's weights."""

import numpy as np

import oracle


def _pack(codes):
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def _bank(q, e_count=1):
    """int4 values [E, N, K] -> packed bank [E, N, K/2] (low nibble first)."""
    q = np.asarray(q, dtype=np.int64) & 0xF
    return (q[..., 0::2] | (q[..., 1::2] << 4)).astype(np.uint8)


def test_block_scale_placement_closed_form():
    r, k, n = 3, 256, 6
    codes = np.full((r, k), 0x2, dtype=np.uint8)           # E2M1 0x2 = 1.0
    rng = np.random.default_rng(0)
    scales = rng.integers(120, 135, (r, k // 32)).astype(np.uint8)
    knz = np.array([5, 40, 100, 127, 130, 255])            # blocks 0, 1, 3, 3, 4, 7
    q = np.zeros((1, n, k), dtype=np.int64)
    q[0, np.arange(n), knz] = [1, -1, 3, 7, -8, 2]
    sw = np.zeros((1, n, k // 128), dtype=np.float32)
    sw[0, :, 0] = [0.5, 0.25, 2.0, 1.0, 0.0, 0.0]
    sw[0, :, 1] = [0.0, 0.0, 0.0, 0.0, 0.125, 4.0]
    got = oracle.grouped_gemm_mxf4_w4(_pack(codes), scales, [0, r], _bank(q), sw)
    for i in range(r):
        for j in range(n):
            kk = knz[j]
            want = (float(sw[0, j, kk // 128]) * float(q[0, j, kk])
                    * 2.0 ** (int(scales[i, kk // 32]) - 127))
            assert got[i, j] == want, (i, j, got[i, j], want)


def test_equals_w4a8_when_block_scales_agree_within_groups():
    rng = np.random.default_rng(1)
    r, k, n, e = 40, 384, 24, 3
    codes = rng.integers(0, 16, (r, k)).astype(np.uint8)
    grp = rng.integers(110, 140, (r, k // 128))
    scales = np.repeat(grp, 4, axis=1).astype(np.uint8)
    vals = np.array([oracle.e2m1_decode(c) for c in range(16)])[codes]
    aq = oracle.e4m3_encode(vals.astype(np.float32))
    assert np.array_equal(oracle.e4m3_decode(aq), vals)   # E2M1 values are e4m3-exact
    as_ = (2.0 ** (grp - 127.0)).astype(np.float32)
    q = rng.integers(-8, 8, (e, n, k))
    sw = rng.uniform(0.002, 0.02, (e, n, k // 128)).astype(np.float32)
    offsets = np.array([0, 15, 15, 40])                    # expert 1 has no rows
    got = oracle.grouped_gemm_mxf4_w4(_pack(codes), scales, offsets, _bank(q), sw)
    ref = oracle.grouped_gemm_w4a8(aq, as_, offsets, _bank(q), sw)
    assert np.array_equal(got, ref)


def test_routing_structure():
    rng = np.random.default_rng(2)
    r, k, n = 10, 128, 8
    codes = rng.integers(0, 16, (r, k)).astype(np.uint8)
    scales = rng.integers(125, 130, (r, k // 32)).astype(np.uint8)
    q = rng.integers(-7, 8, (2, n, k))
    q[1] = -q[0]                                           # expert 1 negates expert 0
    sw = np.ones((2, n, 1), dtype=np.float32)
    offsets = np.array([0, 4, 8])                          # rows 8, 9 belong to no expert
    got = oracle.grouped_gemm_mxf4_w4(_pack(codes), scales, offsets, _bank(q), sw)
    assert np.all(got[8:] == 0.0)
    alt = oracle.grouped_gemm_mxf4_w4(_pack(codes), scales, np.array([0, 8, 8]), _bank(q), sw)
    assert np.array_equal(got[:4], alt[:4])
    assert np.array_equal(got[4:8], -alt[4:8])
