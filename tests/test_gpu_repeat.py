"""Full-size grouped GEMMs run again and again, and at the large layer's shapes.

* The mid layer's gate_up (SwiGLU + requant) and down (bf16) GEMMs on all 32768 routed rows,
  twenty launches in a row on the same operands: every launch must give the same bits, and
  the results meet the parity rules on 256 sampled rows (elementwise GEMM bound for down,
  scales within 1e-4 and at most 0.5% of codes one step apart for the SwiGLU codes).
* The large layer's GEMMs (K=4096, N=3072 and K=1536, N=4096, 131072 routed rows over 128
  Zipf-skewed experts) against the oracle on about 256 sampled rows (from the hottest expert,
  the smallest one and at random) under the same rules.
* The layer's quantizing permutation (fge_moe_permute_quant) against the oracle's G128
  quantization followed by its permutation, bit for bit, at the mid and large sizes."""

import numpy as np
import pytest
import torch

import oracle
from util import abs_grouped, check_gemm, host, to_dev
from workloads import moe_inputs

pytestmark = pytest.mark.gpu


def _rows_subproblem(aq, as_, offsets, rows):
    """The routed rows `rows` (sorted) as their own grouped problem: same experts, offsets
    over the selection."""
    e_of = np.searchsorted(offsets, rows, side="right") - 1
    counts = np.bincount(e_of, minlength=len(offsets) - 1)
    sub_off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return aq[rows], as_[rows], sub_off


def _setup(fge, name):
    inp = moe_inputs(name, seed=0)
    dev = torch.device("cuda:0")
    x = torch.from_numpy(inp.x_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    logits = torch.from_numpy(inp.logits).to(dev)
    ids, _ = fge.moe_topk_gate(logits, inp.k)
    p = fge.moe_permute_quant(ids, inp.E, x)
    w_gu, s_gu = fge.w4_prepack(to_dev(inp.w_gu), to_dev(inp.s_gu), True)
    w_dn, s_dn = fge.w4_prepack(to_dev(inp.w_dn), to_dev(inp.s_dn))
    return inp, ids, x, p, (w_gu, s_gu, w_dn, s_dn)


def _check_gate_up(inp, p_host, hq, hs, rows):
    aq, as_, off = _rows_subproblem(p_host["aq"], p_host["as_"], p_host["offsets"], rows)
    c = oracle.grouped_gemm_w4a8(aq, as_, off, inp.w_gu, inp.s_gu)
    rq, rs, _ = oracle.swiglu_requant(c, inp.I)
    np.testing.assert_allclose(hs[rows], rs, rtol=1e-4)
    diff = hq[rows] != rq
    assert diff.mean() <= 0.005, diff.mean()
    assert np.all(np.abs(hq[rows][diff].astype(int) - rq[diff].astype(int)) == 1)


def _check_down(inp, p_host, hq, hs, y, rows):
    aq, as_, off = _rows_subproblem(hq, hs, p_host["offsets"], rows)
    ref = oracle.grouped_gemm_w4a8(aq, as_, off, inp.w_dn, inp.s_dn)
    absref = abs_grouped(aq, as_, off, inp.w_dn, inp.s_dn)
    check_gemm(y[rows], ref, absref, True)


def test_mid_gemms_twenty_launches_identical_and_in_parity(fge):
    inp, ids, x, p, (w_gu, s_gu, w_dn, s_dn) = _setup(fge, "mid")
    r = inp.T * inp.k
    dev = x.device
    ws = fge.new_workspace(fge.workspace_bytes(fge.OP_GROUPED_GEMM), dev)
    hq = torch.empty((r, inp.I), dtype=torch.uint8, device=dev)
    hs = torch.empty((r, inp.I // 128), dtype=torch.float32, device=dev)
    y = torch.empty((r, inp.H), dtype=torch.bfloat16, device=dev)
    fge.clear_device_status(ws)
    first = None
    for it in range(20):
        fge.grouped_gemm_w4a8(p["aq"], p["as_"], p["offsets"], w_gu, s_gu, epilogue="swiglu",
                              workspace=ws, out=hq, scales=hs)
        fge.grouped_gemm_w4a8(hq, hs, p["offsets"], w_dn, s_dn, out_dtype=torch.bfloat16,
                              workspace=ws, out=y)
        cur = (hq.clone(), hs.clone(), y.clone())
        if first is None:
            first = cur
        else:
            for a, b in zip(first, cur):
                assert torch.equal(a, b), "launch %d differs from the first" % it
    assert fge.read_device_status(ws) == 0
    p_host = {k: host(p[k]) for k in ("aq", "as_", "offsets")}
    rows = np.sort(np.random.default_rng(3).choice(r, size=256, replace=False))
    hq_h, hs_h = host(first[0]), host(first[1])
    _check_gate_up(inp, p_host, hq_h, hs_h, rows)
    _check_down(inp, p_host, hq_h, hs_h, host(first[2]).astype(np.float64), rows)


def test_large_shape_gemms_on_sampled_rows(fge):
    inp, ids, x, p, (w_gu, s_gu, w_dn, s_dn) = _setup(fge, "large")
    hq, hs = fge.grouped_gemm_w4a8(p["aq"], p["as_"], p["offsets"], w_gu, s_gu,
                                   epilogue="swiglu")
    y = fge.grouped_gemm_w4a8(hq, hs, p["offsets"], w_dn, s_dn, out_dtype=torch.bfloat16)
    p_host = {k: host(p[k]) for k in ("aq", "as_", "offsets")}
    off = p_host["offsets"]
    counts = np.diff(off)
    # Zipf-skewed routing: the hottest expert far above the mean, the coldest nearly empty
    assert counts.max() > 10 * counts.mean() and counts.min() < counts.mean() / 100
    rng = np.random.default_rng(4)
    # rows of the hottest expert, of the smallest non-empty one, and random ones
    hot = int(np.argmax(counts))
    small = int(np.argmin(np.where(counts > 0, counts, counts.max() + 1)))
    rows = np.unique(np.concatenate([
        rng.choice(np.arange(off[hot], off[hot + 1]), 64, replace=False),
        np.arange(off[small], off[small + 1])[:32],
        rng.choice(inp.T * inp.k, 160, replace=False)]))
    hq_h, hs_h = host(hq), host(hs)
    _check_gate_up(inp, p_host, hq_h, hs_h, rows)
    _check_down(inp, p_host, hq_h, hs_h, host(y).astype(np.float64), rows)


@pytest.mark.parametrize("name", ["mid", "large"])
def test_quantizing_permutation_matches_the_oracle(fge, name):
    inp = moe_inputs(name, seed=0)
    dev = torch.device("cuda:0")
    x = torch.from_numpy(inp.x_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    ids, _ = fge.moe_topk_gate(torch.from_numpy(inp.logits).to(dev), inp.k)
    got = fge.moe_permute_quant(ids, inp.E, x)
    xq, xs = oracle.quant_act_g128(inp.x)
    ref = oracle.moe_permute(host(ids), inp.E, xq, xs)
    for key in ("offsets", "row_token", "token_row", "aq"):
        assert np.array_equal(host(got[key]), ref[key]), key
    assert np.array_equal(host(got["as_"]).view(np.uint32), ref["as_"].view(np.uint32))
