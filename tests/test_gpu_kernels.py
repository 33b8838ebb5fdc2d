"""GPU parity of the memory-bound kernels against the CPU oracle, through the C ABI:
activation quant (bit-exact codes and scales), top-k gate (exact ids, gates to 2e-6),
permutation (bit-exact), combine and the unfused SwiGLU requant."""

import numpy as np
import pytest
import torch

import oracle
from util import bf16_dev, bf16_ulp, host, to_dev
from workloads import moe_inputs, to_bf16

pytestmark = pytest.mark.gpu


def _x(m, k, seed, kind="normal"):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((m, k)).astype(np.float32)
    if kind == "mixed":
        x[0] = 0.0                                          # all-zero row
        if m > 1:
            x[1] *= np.float32(1e-30)                       # tiny row
        if m > 2:
            x[2, ::7] *= np.float32(300.0)                  # outliers
        x *= np.exp(rng.uniform(-4, 4, (m, 1))).astype(np.float32)
    return to_bf16(x)


@pytest.mark.parametrize("m,k", [(1, 128), (3, 256), (300, 2560), (64, 4096), (1000, 2048)])
def test_quant_g128_bit_exact(fge, m, k):
    bits, xv = _x(m, k, seed=m + k, kind="mixed")
    xq, xs = fge.fp8_quant_act(bf16_dev(bits), "g128")
    rq, rs = oracle.quant_act_g128(xv)
    assert np.array_equal(host(xq), rq)
    assert np.array_equal(host(xs), rs)


@pytest.mark.parametrize("m,k", [(1, 2560), (16, 2560), (300, 2560), (2048, 2560)])
def test_quant_per_tensor_bit_exact(fge, m, k):
    bits, xv = _x(m, k, seed=7 * m)
    xq, xs = fge.fp8_quant_act(bf16_dev(bits), "tensor")
    rq, rs = oracle.quant_act_per_tensor(xv)
    assert host(xs)[0] == rs
    assert np.array_equal(host(xq), rq)


def test_quant_zero_input_scale_floor(fge):
    z = torch.zeros((16, 256), dtype=torch.bfloat16, device="cuda")
    xq, xs = fge.fp8_quant_act(z, "tensor")
    assert host(xs)[0] == 1.0 and not host(xq).any()
    xq, xs = fge.fp8_quant_act(z, "g128")
    assert np.all(host(xs) == 1.0) and not host(xq).any()


@pytest.mark.parametrize("t,e,k", [(64, 8, 2), (4096, 64, 8), (1000, 128, 8), (33, 256, 32),
                                   (500, 96, 8), (300, 100, 6), (257, 40, 32), (77, 1000, 16)])
def test_topk_gate(fge, t, e, k):
    rng = np.random.default_rng(t + e)
    lg = rng.standard_normal((t, e)).astype(np.float32)
    lg[: t // 4] = np.round(lg[: t // 4] * 2) / 2            # many exact ties
    ids, gates = fge.moe_topk_gate(to_dev(lg), k)
    rid, rg = oracle.topk_gate(lg, k)
    assert np.array_equal(host(ids), rid)
    np.testing.assert_allclose(host(gates), rg, rtol=2e-6, atol=0)


def test_topk_gate_signed_zeros_tie(fge):
    # -0 and +0 are equal logits: among them the lower expert id is taken first
    rng = np.random.default_rng(5)
    lg = np.where(rng.random((256, 64)) < 0.5, np.float32(-0.0), np.float32(0.0))
    lg[:, 40] = -1.0
    lg[::3, 7] = 2.0
    ids, gates = fge.moe_topk_gate(to_dev(lg.astype(np.float32)), 4)
    rid, rg = oracle.topk_gate(lg.astype(np.float32), 4)
    assert np.array_equal(host(ids), rid)
    np.testing.assert_allclose(host(gates), rg, rtol=2e-6, atol=0)


@pytest.mark.parametrize("t,e,k,h", [(64, 8, 2, 256), (4096, 64, 8, 2048), (333, 128, 8, 512),
                                     (200, 16, 1, 128), (1000, 256, 3, 256), (129, 32, 5, 128)])
def test_permute_bit_exact(fge, t, e, k, h):
    rng = np.random.default_rng(t * k)
    bias = -1.1 * np.log(np.arange(1, e + 1))                  # skewed: some experts empty
    lg = (rng.standard_normal((t, e)) + bias).astype(np.float32)
    ids, _ = oracle.topk_gate(lg, k)
    xq = rng.integers(0, 256, size=(t, h), dtype=np.uint8)
    xs = rng.uniform(0.001, 1, size=(t, h // 128)).astype(np.float32)
    got = fge.moe_permute(to_dev(ids), e, to_dev(xq), to_dev(xs))
    ref = oracle.moe_permute(ids, e, xq, xs)
    for key in ["offsets", "row_token", "token_row", "aq", "as_"]:
        assert np.array_equal(host(got[key]), ref[key]), key


@pytest.mark.parametrize("y_dtype,out_dtype", [(torch.float32, torch.float32),
                                               (torch.bfloat16, torch.bfloat16),
                                               (torch.float32, torch.bfloat16)])
def test_combine(fge, y_dtype, out_dtype):
    rng = np.random.default_rng(5)
    t, e, k, h = 300, 16, 4, 640
    ids, gates = oracle.topk_gate(rng.standard_normal((t, e)).astype(np.float32), k)
    p = oracle.moe_permute(ids, e, np.zeros((t, 128), np.uint8), np.zeros((t, 1), np.float32))
    y = rng.standard_normal((t * k, h)).astype(np.float32)
    if y_dtype == torch.bfloat16:
        y = to_bf16(y)[1]
    out = fge.moe_combine(to_dev(y).to(y_dtype), to_dev(p["token_row"]), to_dev(gates),
                          out_dtype=out_dtype)
    ref = oracle.moe_combine(y, p["token_row"], gates)
    got = host(out).astype(np.float64)
    if out_dtype == torch.float32:
        np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-6)
    else:
        # one bf16 ulp of the result plus the fp32 accumulation error of the k terms
        absref = oracle.moe_combine(np.abs(y), p["token_row"], gates)
        assert np.all(np.abs(got - ref) <= bf16_ulp(ref) + 1e-6 * absref)


@pytest.mark.parametrize("t,e,k,h,out_dtype", [(333, 64, 8, 2048, torch.bfloat16),
                                               (97, 16, 1, 4096, torch.bfloat16),
                                               (1000, 32, 3, 2048, torch.float32),
                                               (1, 8, 8, 6144, torch.bfloat16)])
def test_combine_staged_equals_plain(fge, t, e, k, h, out_dtype):
    # the layer's combine (slot rows staged in shared memory by bulk copies) gives the plain
    # kernel's bits, and meets the oracle's rule
    rng = np.random.default_rng(t + h)
    ids, gates = oracle.topk_gate(rng.standard_normal((t, e)).astype(np.float32), k)
    p = oracle.moe_permute(ids, e, np.zeros((t, 128), np.uint8), np.zeros((t, 1), np.float32))
    y = to_bf16(rng.standard_normal((t * k, h)).astype(np.float32))[1]
    yd, tr, gd = to_dev(y).to(torch.bfloat16), to_dev(p["token_row"]), to_dev(gates)
    ws = fge.new_workspace(256, yd.device)
    fge.clear_device_status(ws)
    staged = fge.moe_combine(yd, tr, gd, out_dtype=out_dtype, workspace=ws)
    plain = fge.moe_combine(yd, tr, gd, out_dtype=out_dtype)
    assert fge.read_device_status(ws) == 0
    assert torch.equal(staged, plain)
    ref = oracle.moe_combine(y, p["token_row"], gates)
    absref = oracle.moe_combine(np.abs(y), p["token_row"], gates)
    got = host(staged).astype(np.float64)
    ulp = bf16_ulp(ref) if out_dtype == torch.bfloat16 else 1e-6 * np.abs(ref)
    assert np.all(np.abs(got - ref) <= ulp + 1e-6 * absref)


def test_combine_staged_refusals(fge):
    t, k, h = 16, 2, 2048
    y = torch.zeros((t * k, h), dtype=torch.bfloat16, device="cuda")
    tr = torch.zeros((t, k), dtype=torch.int32, device="cuda")
    g = torch.zeros((t, k), dtype=torch.float32, device="cuda")
    ws = fge.new_workspace(256, y.device)
    with pytest.raises(fge.FgeError):           # H not a multiple of 2048
        fge.moe_combine(y[:, :1024].contiguous(), tr, g, workspace=ws)
    big = torch.zeros((t, 9), dtype=torch.int32, device="cuda")
    with pytest.raises(fge.FgeError):           # k > 8
        fge.moe_combine(torch.zeros((t * 9, h), dtype=torch.bfloat16, device="cuda"), big,
                        torch.zeros((t, 9), dtype=torch.float32, device="cuda"), workspace=ws)
    with pytest.raises(fge.FgeError):           # the workspace holds no status header
        fge.moe_combine(y, tr, g, workspace=fge.new_workspace(256, y.device)[:128])


def test_swiglu_quant_unfused(fge):
    rng = np.random.default_rng(6)
    r, inter = 500, 768
    c = (rng.standard_normal((r, 2 * inter)) * 4).astype(np.float32)
    hq, hs = fge.swiglu_quant(to_dev(c), inter)
    rq, rs, _ = oracle.swiglu_requant(c, inter)
    gq, gs = host(hq), host(hs)
    np.testing.assert_allclose(gs, rs, rtol=1e-5)
    diff = gq != rq
    assert diff.mean() <= 0.005, diff.mean()
    # where codes differ they are neighbours (one e4m3 step, same sign)
    d = np.abs(gq[diff].astype(int) - rq[diff].astype(int))
    assert np.all(d == 1)


def test_tiny_inputs_layer_routing_consistency(fge):
    inp = moe_inputs("tiny", seed=2)
    ids, gates = fge.moe_topk_gate(to_dev(inp.logits), inp.k)
    rid, _ = oracle.topk_gate(inp.logits, inp.k)
    assert np.array_equal(host(ids), rid)


@pytest.mark.parametrize("t,e,k,h", [(64, 8, 2, 256), (4096, 64, 8, 2048), (333, 128, 3, 384)])
def test_permute_quant_equals_quant_then_permute(fge, t, e, k, h):
    """The quantization folded into the permutation gives exactly the codes, scales and
    indices of quantizing first and permuting after."""
    rng = np.random.default_rng(t + 3 * k)
    lg = rng.standard_normal((t, e)).astype(np.float32)
    x = (rng.standard_normal((t, h)) * np.exp(rng.uniform(-4, 4, (t, 1)))).astype(np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    xd = bf16_dev(bits)
    ids, _ = fge.moe_topk_gate(to_dev(lg), k)
    xq, xs = fge.fp8_quant_act(xd, "g128")
    a = fge.moe_permute(ids, e, xq, xs)
    b = fge.moe_permute_quant(ids, e, xd)
    for key in ("offsets", "row_token", "token_row", "aq", "as_"):
        assert torch.equal(a[key], b[key]), key
