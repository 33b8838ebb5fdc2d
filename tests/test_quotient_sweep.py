"""Host check of the quotient the GPU activation quantizers use (csrc/quotient.cuh): one
correctly rounded reciprocal per scale, the product, and one exact-residual correction give
the IEEE float32 quotient x / s for every bfloat16 x and normal float32 s.  The C program
runs on every 16th significand of s here (every one was checked once: 2^30 pairs, none
differ); the plain reciprocal product must differ on some pairs, so the check can fail."""

import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def _run(tmp_path, *args):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "quotient_sweep")
    subprocess.run([cc, "-O2", "-ffp-contract=off", "-o", exe,
                    os.path.join(HERE, "host", "quotient_sweep.c"), "-lm"], check=True)
    out = subprocess.run([exe, *args], check=True, capture_output=True, text=True).stdout
    pairs, bad = out.split()[1], out.split()[3]
    return int(pairs), int(bad)


def test_corrected_quotient_equals_the_division(tmp_path):
    pairs, bad = _run(tmp_path, "16")
    assert pairs == 128 * (1 << 23) // 16
    assert bad == 0


def test_plain_reciprocal_product_is_not_the_division(tmp_path):
    pairs, bad = _run(tmp_path, "16", "plain")
    assert bad > 0



@pytest.mark.parametrize("mode", ["amax", "wide"])
def test_corrected_quotient_across_exponents(tmp_path, mode):
    # random bf16 x (zeros, subnormals, both signs) and s across the range the kernels take
    # the reciprocal path for: the e4m3 codes of the two quotients agree everywhere
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "quotient_range")
    subprocess.run([cc, "-O2", "-ffp-contract=off", "-o", exe,
                    os.path.join(HERE, "host", "quotient_range.c"), "-lm"], check=True)
    out = subprocess.run([exe, "2000000", "7", mode], check=True, capture_output=True,
                         text=True).stdout.split()
    assert int(out[1]) == 2000000 and int(out[3]) == 0


def test_group_scale_by_constant_reciprocal(tmp_path):
    # every finite bf16 amax: max(RN(amax / 448), 2^-126) from RN(1/448) and the correction
    # step equals the one from the division
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "quotient_range")
    subprocess.run([cc, "-O2", "-ffp-contract=off", "-o", exe,
                    os.path.join(HERE, "host", "quotient_range.c"), "-lm"], check=True)
    out = subprocess.run([exe, "0", "0", "scale"], check=True, capture_output=True,
                         text=True).stdout.split()
    assert int(out[1]) == 0x7F80 and int(out[3]) == 0
