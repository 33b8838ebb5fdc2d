"""MXFP4 activation quantization on the GPU against the oracle, byte for byte."""

import numpy as np
import pytest
import torch

from oracle.mx import MX_BLOCK, mx_quant_e2m1
from util import bf16_dev

pytestmark = pytest.mark.gpu


def _bf16_bits_to_f64(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def _run(fge, bits):
    xq, xs = fge.mx_quant_e2m1(bf16_dev(bits))
    torch.cuda.synchronize()
    return xq.cpu().numpy(), xs.cpu().numpy()


def _check(fge, bits):
    xq, xs = _run(fge, bits)
    rq, rs = mx_quant_e2m1(_bf16_bits_to_f64(bits))
    np.testing.assert_array_equal(xs, rs)
    np.testing.assert_array_equal(xq, rq)


@pytest.mark.parametrize("m,k", [(1, 32), (33, 2048), (7, 96), (129, 256)])
def test_random_rows(fge, m, k):
    rng = np.random.default_rng(m * 1000 + k)
    x = rng.standard_normal((m, k)) * np.exp(rng.uniform(-20, 20, size=(m, 1)))
    x[:, ::17] *= 40.0                                   # outlier columns
    x[0, : min(k, 64)] = 0.0                             # an all-zero block (and a half)
    bits = (torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
            .view(torch.int16).numpy().view(np.uint16))
    _check(fge, bits)


def test_every_bf16_value_in_every_binade(fge):
    """Each finite nonzero normal bf16 value v, in blocks whose scale puts v / 2^E in each of
    [4, 8), [2, 4), [1, 2), [0.5, 1), [0.25, 0.5) and [0.125, 0.25): all rounding cases,
    ties, saturation and underflow to a signed zero."""
    rows = []
    for b in range(-126, 128):                           # binade: |v| in [2^b, 2^(b+1))
        e_field = b + 127
        mags = (e_field << 7) | np.arange(128, dtype=np.uint32)
        vals = np.concatenate([mags, mags | 0x8000]).astype(np.uint16)   # both signs
        for d in range(6):
            if b + d > 127:
                continue
            anchor = np.uint16(((b + d + 127) << 7) if d > 0 else (e_field << 7))
            for i in range(0, len(vals), MX_BLOCK - 1):
                blk = vals[i:i + MX_BLOCK - 1]
                row = np.full(MX_BLOCK, anchor, dtype=np.uint16)
                row[1:1 + len(blk)] = blk
                rows.append(row)
    bits = np.stack(rows)                                # [blocks, 32]
    pad = (-len(bits)) % 64                              # rows of 64 blocks
    bits = np.concatenate([bits, np.zeros((pad, MX_BLOCK), dtype=np.uint16)])
    _check(fge, bits.reshape(-1, 64 * MX_BLOCK))


def test_subnormal_and_sorted_bf16(fge):
    """Every finite bf16 bit pattern, sorted by magnitude, in blocks of 32 (subnormals and
    zeros included)."""
    allb = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = ((allb >> 7) & 0xFF) != 0xFF
    vals = allb[finite]
    order = np.argsort(np.abs(_bf16_bits_to_f64(vals)), kind="stable")
    vals = vals[order]
    pad = (-len(vals)) % (MX_BLOCK * 64)
    vals = np.concatenate([vals, np.zeros(pad, dtype=np.uint16)])
    _check(fge, vals.reshape(-1, MX_BLOCK * 64))


def test_rejects_bad_shape(fge):
    x = torch.zeros((4, 48), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(RuntimeError):
        fge.mx_quant_e2m1(x)
