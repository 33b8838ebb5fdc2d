"""The premise of the G128 quantizers' amax: over bfloat16 values, the low 15 bits of the
pattern order like the magnitude, so an unsigned maximum of (w & 0x7fff) picks the pattern
of the largest |x| (zeros of either sign and subnormals included), and the patterns at or
above 0x7f80 are exactly the infinities and NaNs.  Checked over all 2^16 patterns with the
values decoded by numpy, not by the bit rule."""
import numpy as np
import pytest

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _values():
    bits = np.arange(1 << 16, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    return bits, vals


def test_nonfinite_patterns_are_exactly_the_top_magnitudes():
    bits, vals = _values()
    mag = bits & 0x7FFF
    assert np.array_equal(mag >= 0x7F80, ~np.isfinite(vals))


def test_magnitude_bits_order_like_the_absolute_value():
    bits, vals = _values()
    fin = np.isfinite(vals)
    mag = (bits & 0x7FFF)[fin]
    a = np.abs(vals[fin].astype(np.float64))
    order = np.argsort(mag, kind="stable")
    # strictly increasing bits give non-decreasing magnitudes, and equal magnitudes (only
    # +0 and -0) share one masked pattern
    assert np.all(np.diff(a[order]) >= 0)
    for m in np.unique(mag):
        assert np.unique(a[mag == m]).size == 1


def test_masked_maximum_equals_float_maximum_on_random_groups():
    rng = np.random.default_rng(5)
    bits, vals = _values()
    finite = bits[np.isfinite(vals)]
    for _ in range(2000):
        g = rng.choice(finite, size=128).astype(np.uint32)
        m = int((g & 0x7FFF).max())
        amax = np.float32(np.uint32(m << 16).view(np.float32))
        ref = np.abs((g << 16).view(np.float32)).max()
        assert amax == ref and not np.signbit(amax)
