"""Both CPU oracles against e4m3 codes worked out by hand (tests/golden/, cited there)."""

import numpy as np

import oracle
from golden_data import e4m3_points
from oracle import native


def test_fixture_is_nontrivial():
    pts = e4m3_points()
    assert len(pts) >= 20
    assert {c for _, c, _ in pts} >= {0x00, 0x01, 0x7E, 0x80}


def test_numpy_oracle_encodes_hand_derived_points():
    pts = e4m3_points()
    x = np.array([v for v, _, _ in pts], np.float32)
    want = np.array([c for _, c, _ in pts], np.uint8)
    assert np.array_equal(oracle.e4m3_encode(x), want)


def test_cpp_oracle_encodes_hand_derived_points():
    pts = e4m3_points()
    x = np.array([v for v, _, _ in pts], np.float32)
    want = np.array([c for _, c, _ in pts], np.uint8)
    assert np.array_equal(native.e4m3_encode(x), want)


def test_decode_of_hand_derived_codes():
    # every finite point that is itself an e4m3 value decodes back to it
    mags = set(oracle.e4m3_decode_table()[:0x7F].tolist())
    for v, c, _ in e4m3_points():
        if abs(v) in mags:
            assert oracle.e4m3_decode(np.uint8(c)) == np.float64(v)
            assert native.e4m3_decode_table()[c] == np.float64(v)
