"""The GPU quantizers on inputs whose e4m3 code hangs on the last bits of x / s.

The code of an activation is the e4m3 rounding of the float32 quotient x / s.  A quantizer
that multiplied by a rounded reciprocal instead would be off by one code step whenever a
point halfway between two e4m3 values falls between x * fl(1/s) and fl(x / s).  These
inputs are exactly such (x, amax) pairs, found by searching every finite bfloat16 x against
seeded bfloat16 amax values.  Each 128-value group holds its amax (so s = amax / 448 as the
oracle forms it) and up to 127 such x; every quantizer that feeds the path (G128 alone, G128
inside the permuted copy, per-row, per-tensor) must give the oracle's codes bit for bit.
"""

import functools

import numpy as np
import pytest
import torch

import oracle
from util import DEV

pytestmark = pytest.mark.gpu


@functools.lru_cache(maxsize=None)
def _hard_pairs(n_amax=400, seed=7):
    """(amax, [x ...]) for which the product rule and the quotient rule disagree."""
    rng = np.random.default_rng(seed)
    bits = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    xs = bits[np.isfinite(bits)]
    out = []
    for a in ((rng.integers(0x3A00, 0x4500, n_amax).astype(np.uint32) << 16).view(np.float32)):
        x = xs[np.abs(xs) <= a]
        s = np.float32(a) / np.float32(448.0)
        prod = (x * (np.float32(1.0) / s)).astype(np.float32)
        quot = (x / s).astype(np.float32)
        diff = oracle.e4m3_encode(prod) != oracle.e4m3_encode(quot)
        if diff.any():
            out.append((np.float32(a), x[diff]))
    return out


@pytest.fixture(scope="module")
def hard_rows():
    """Rows of 128-value groups: group = [amax, up to 127 hard x of that amax, zeros]."""
    groups = []
    for a, xh in _hard_pairs():
        for i in range(0, len(xh), 127):
            g = np.zeros(128, np.float32)
            g[0] = a
            part = xh[i:i + 127]
            g[1:1 + len(part)] = part
            groups.append(g)
    assert len(groups) >= 8, "the search found too few disagreeing pairs to test anything"
    n = (len(groups) + 3) // 4 * 4
    while len(groups) < n:
        groups.append(np.zeros(128, np.float32))
    rows = np.stack(groups).reshape(n // 4, 512)   # 4 groups per row (K = 512)
    return rows, sum(len(xh) for _, xh in _hard_pairs())


def _bf16(rows):
    x = torch.from_numpy(rows).to(torch.bfloat16)
    assert np.array_equal(x.float().numpy(), rows)   # every value is bf16-exact
    return x.to(DEV)


def test_g128_codes_on_hard_quotients(fge, hard_rows):
    rows, n_hard = hard_rows
    assert n_hard > 100
    xq, xs = fge.fp8_quant_act(_bf16(rows), "g128")
    q_ref, s_ref = oracle.quant_act_g128(rows)
    assert np.array_equal(xs.cpu().numpy(), s_ref)
    assert np.array_equal(xq.cpu().numpy(), q_ref)


def test_permute_quant_codes_on_hard_quotients(fge, hard_rows):
    rows, _ = hard_rows
    t = rows.shape[0]
    rng = np.random.default_rng(3)
    ids = np.stack([rng.choice(8, 2, replace=False) for _ in range(t)]).astype(np.int32)
    p = fge.moe_permute_quant(torch.from_numpy(ids).to(DEV), 8, _bf16(rows))
    q_ref, s_ref = oracle.quant_act_g128(rows)
    ref = oracle.moe_permute(ids, 8, q_ref, s_ref)
    assert np.array_equal(p["aq"].cpu().numpy(), ref["aq"])
    assert np.array_equal(p["as_"].cpu().numpy(), ref["as_"])


def test_per_row_codes_on_hard_quotients(fge, hard_rows):
    rows, _ = hard_rows
    # one group per row, so each row's amax is its group's amax
    r1 = rows.reshape(-1, 128)
    xq, xs = fge.fp8_quant_act(_bf16(r1), "row")
    q_ref, s_ref = oracle.quant_act_per_row(r1)
    assert np.array_equal(xs.cpu().numpy(), s_ref)
    assert np.array_equal(xq.cpu().numpy(), q_ref)


def test_per_tensor_codes_on_hard_quotients(fge):
    # per-tensor: one tensor per amax, for the amax values with the most disagreeing pairs
    pairs = sorted(_hard_pairs(), key=lambda p: -len(p[1]))[:4]
    for a, xh in pairs:
        k = (len(xh) + 1 + 127) // 128 * 128
        row = np.zeros(k, np.float32)
        row[0] = a
        row[1:1 + len(xh)] = xh
        xq, xs = fge.fp8_quant_act(_bf16(row[None, :]), "tensor")
        q_ref, s_ref = oracle.quant_act_per_tensor(row[None, :])
        assert float(xs.cpu().numpy()[0]) == float(s_ref)
        assert np.array_equal(xq.cpu().numpy(), q_ref)


def _tiny_rows(seed):
    """Groups whose scale falls on either side of 2^-90 (below it the quantizers divide, above
    it they use the reciprocal and the correction), holding subnormal bfloat16 values, signed
    zeros and values across the group's whole range."""
    rng = np.random.default_rng(seed)
    groups = []
    for e_amax in (-120, -100, -82, -81, -80, -60, -20, 0, 20, 100, 127):
        g = rng.uniform(-1.0, 1.0, 128).astype(np.float32) * np.float32(2.0 ** e_amax)
        g[0] = np.float32(2.0 ** e_amax) * np.float32(1.5)            # the group's amax
        g[1:9] = np.float32(2.0 ** -133) * np.arange(1, 9)            # bf16 subnormals
        g[9], g[10] = np.float32(0.0), np.float32(-0.0)
        g[11:20] *= -1
        groups.append(torch.from_numpy(g).to(torch.bfloat16).float().numpy())
    while len(groups) % 4:
        groups.append(np.zeros(128, np.float32))
    return np.stack(groups).reshape(-1, 512)


def test_quantizers_across_the_reciprocal_range(fge):
    rows = _tiny_rows(11)
    xq, xs = fge.fp8_quant_act(_bf16(rows), "g128")
    q_ref, s_ref = oracle.quant_act_g128(rows)
    assert np.array_equal(xs.cpu().numpy(), s_ref)
    assert np.array_equal(xq.cpu().numpy(), q_ref)
    r1 = rows.reshape(-1, 128)
    xq, xs = fge.fp8_quant_act(_bf16(r1), "row")
    q_ref, s_ref = oracle.quant_act_per_row(r1)
    assert np.array_equal(xs.cpu().numpy(), s_ref)
    assert np.array_equal(xq.cpu().numpy(), q_ref)
    for g in r1:                                      # each group as its own tensor
        xq, xs = fge.fp8_quant_act(_bf16(g[None, :]), "tensor")
        q_ref, s_ref = oracle.quant_act_per_tensor(g[None, :])
        assert float(xs.cpu().numpy()[0]) == float(s_ref)
        assert np.array_equal(xq.cpu().numpy(), q_ref)
