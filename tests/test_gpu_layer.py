"""End-to-end MoE layer parity (one C-ABI call: gate -> quant -> permute -> gate_up with
fused SwiGLU requant -> down -> combine) against the oracle: cosine >= 0.9999.

The layer is row-independent (routing, quantization and every expert GEMM act per token),
so at the full mid and large sizes the GPU runs the whole layer and the oracle recomputes a
seeded sample of tokens on its own; the sampled rows of the GPU output must match."""

import numpy as np
import pytest
import torch

import oracle
from oracle import native
from util import bf16_dev, cosine, host, to_dev
from workloads import moe_inputs

pytestmark = pytest.mark.gpu


def _run_layer(fge, inp, fmt):
    w_gu, s_gu = fge.w4_prepack(to_dev(inp.w_gu), to_dev(inp.s_gu), gate_up_interleave=True,
                                fmt=fmt)
    w_dn, s_dn = fge.w4_prepack(to_dev(inp.w_dn), to_dev(inp.s_dn), fmt=fmt)
    od = torch.float32 if inp.out == "f32" else torch.bfloat16
    out = fge.moe_layer_forward(to_dev(inp.logits), bf16_dev(inp.x_bits), inp.k, inp.I, w_gu,
                                s_gu, w_dn, s_dn, fmt=fmt, out_dtype=od)
    torch.cuda.synchronize()
    return host(out)


def _oracle_rows(inp, rows):
    out, _ = oracle.moe_layer_forward(inp.logits[rows], inp.x[rows], inp.k, inp.w_gu, inp.s_gu,
                                      inp.w_dn, inp.s_dn, inp.I, out_dtype=inp.out)
    return out


@pytest.mark.parametrize("fmt_name", ["lut", "subnormal"])
def test_tiny_layer(fge, fmt_name):
    fmt = fge.W4_LUT if fmt_name == "lut" else fge.W4_SUBNORMAL
    inp = moe_inputs("tiny", seed=11)
    got = _run_layer(fge, inp, fmt)
    ref = _oracle_rows(inp, np.arange(inp.T))
    assert cosine(got, ref) >= 0.9999
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel < 5e-3, rel
    # the single-threaded C++ oracle restates the same layer independently
    ref_c = native.moe_layer_forward(inp.logits, inp.x, inp.k, inp.w_gu, inp.s_gu, inp.w_dn,
                                     inp.s_dn, inp.I, out_dtype=inp.out)
    assert cosine(got, ref_c) >= 0.9999


@pytest.mark.parametrize("name,sample", [("mid", 384), ("large", 160)])
def test_full_size_layer_sampled(fge, name, sample):
    inp = moe_inputs(name, seed=0)
    if name == "large":
        counts = np.bincount(oracle.topk_gate(inp.logits[:2048], inp.k)[0].ravel(),
                             minlength=inp.E)
        assert counts.max() > 10 * counts.mean() and (counts == 0).any()
    got = _run_layer(fge, inp, fge.W4_SUBNORMAL)
    rows = np.sort(np.random.default_rng(5).choice(inp.T, size=sample, replace=False))
    ref = _oracle_rows(inp, rows)
    assert np.all(np.isfinite(got))
    c = cosine(got[rows], ref)
    assert c >= 0.9999, c


def test_host_pipeline_matches_layer_calls(fge):
    """HostLayerPipeline: three steps with different inputs, from pinned host buffers to
    pinned host buffers with the copies overlapped, equal the plain layer calls bit for bit
    (same kernels; the slots alternate between steps), with and without CUDA graphs."""
    inp = moe_inputs("tiny", seed=5)
    w_gu, s_gu = fge.w4_prepack(to_dev(inp.w_gu), to_dev(inp.s_gu), gate_up_interleave=True)
    w_dn, s_dn = fge.w4_prepack(to_dev(inp.w_dn), to_dev(inp.s_dn))
    rng = np.random.default_rng(9)
    xs, lgs, refs, outs = [], [], [], []
    for i in range(3):
        x = bf16_dev(inp.x_bits) * (1.0 + i)
        lg = to_dev(inp.logits) + to_dev(rng.standard_normal(inp.logits.shape).astype(np.float32))
        refs.append(host(fge.moe_layer_forward(lg, x, inp.k, inp.I, w_gu, s_gu, w_dn, s_dn)))
        xs.append(x.cpu().pin_memory())
        lgs.append(lg.cpu().pin_memory())
        outs.append(torch.empty((inp.T, inp.H), dtype=torch.bfloat16).pin_memory())
    torch.cuda.synchronize()
    for graphs in (False, True):
        pipe = fge.HostLayerPipeline(inp.T, inp.H, inp.E, inp.k, inp.I, w_gu, s_gu, w_dn, s_dn,
                                     graphs=graphs)
        for o in outs:
            o.zero_()
        for i in range(3):
            pipe.submit(xs[i], lgs[i], outs[i])
        pipe.finish()
        for i in range(3):
            np.testing.assert_array_equal(outs[i].float().numpy(), refs[i])


@pytest.mark.parametrize("name,t", [("mid", 4096), ("large", 1536)])
def test_layer_equals_its_stage_calls(fge, name, t):
    """The layer call (whose combine at H % 2048 == 0 runs on bulk copies into shared memory)
    equals the same stages called one by one through the C ABI, ending with the plain
    combine kernel of fge_moe_combine, bit for bit."""
    inp = moe_inputs(name, seed=3, T=t)
    w_gu, s_gu = fge.w4_prepack(to_dev(inp.w_gu), to_dev(inp.s_gu), gate_up_interleave=True)
    w_dn, s_dn = fge.w4_prepack(to_dev(inp.w_dn), to_dev(inp.s_dn))
    lg, x = to_dev(inp.logits), bf16_dev(inp.x_bits)
    layer = host(fge.moe_layer_forward(lg, x, inp.k, inp.I, w_gu, s_gu, w_dn, s_dn))
    ids, gates = fge.moe_topk_gate(lg, inp.k)
    p = fge.moe_permute_quant(ids, inp.E, x)
    hq, hs = fge.grouped_gemm_w4a8(p["aq"], p["as_"], p["offsets"], w_gu, s_gu,
                                   epilogue="swiglu")
    y = fge.grouped_gemm_w4a8(hq, hs, p["offsets"], w_dn, s_dn, out_dtype=torch.bfloat16)
    staged = host(fge.moe_combine(y, p["token_row"], gates))
    torch.cuda.synchronize()
    assert np.all(np.isfinite(layer))
    np.testing.assert_array_equal(layer, staged)
