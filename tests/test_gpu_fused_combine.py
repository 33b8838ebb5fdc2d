"""The MoE layer with the combine folded into the down GEMM's epilogue
(fge_moe_layer_forward_fused_combine).

The last of a token's k slot rows to land combines the token's chunk in slot order with the
combine kernel's own fmaf chain, so the fused layer must equal the plain layer (bf16 output)
bit for bit, whatever order the tiles ran in, and both must meet the layer rule against the
oracle.  Cases: the tiny layer (both bank formats), the mid layer twice over, and a
2048-token prefix of the large skewed layer (hot experts far above the mean, some experts
with no rows)."""

import numpy as np
import pytest
import torch

import oracle
from util import bf16_dev, cosine, host, to_dev
from workloads import moe_inputs

pytestmark = pytest.mark.gpu


def _banks(fge, inp, fmt):
    w_gu, s_gu = fge.w4_prepack(to_dev(inp.w_gu), to_dev(inp.s_gu), gate_up_interleave=True,
                                fmt=fmt)
    w_dn, s_dn = fge.w4_prepack(to_dev(inp.w_dn), to_dev(inp.s_dn), fmt=fmt)
    return w_gu, s_gu, w_dn, s_dn


def _both(fge, logits, x_bits, inp, banks, fmt, repeats=1):
    lg, x = to_dev(logits), bf16_dev(x_bits)
    plain = host(fge.moe_layer_forward(lg, x, inp.k, inp.I, *banks, fmt=fmt))
    fused = []
    for _ in range(repeats):
        fused.append(host(fge.moe_layer_forward(lg, x, inp.k, inp.I, *banks, fmt=fmt,
                                                fused_combine=True)))
    torch.cuda.synchronize()
    return plain, fused


@pytest.mark.parametrize("fmt_name", ["lut", "subnormal"])
def test_tiny_fused_equals_plain_and_oracle(fge, fmt_name):
    fmt = fge.W4_LUT if fmt_name == "lut" else fge.W4_SUBNORMAL
    inp = moe_inputs("tiny", seed=11)
    plain, fused = _both(fge, inp.logits, inp.x_bits, inp, _banks(fge, inp, fmt), fmt)
    assert np.array_equal(fused[0], plain)
    ref, _ = oracle.moe_layer_forward(inp.logits, inp.x, inp.k, inp.w_gu, inp.s_gu, inp.w_dn,
                                      inp.s_dn, inp.I, out_dtype="bf16")
    assert cosine(fused[0], ref) >= 0.9999


def test_mid_fused_equals_plain_repeatedly(fge):
    inp = moe_inputs("mid", seed=0)
    plain, fused = _both(fge, inp.logits, inp.x_bits, inp, _banks(fge, inp, fge.W4_SUBNORMAL),
                         fge.W4_SUBNORMAL, repeats=3)
    assert np.all(np.isfinite(plain))
    for f in fused:
        assert np.array_equal(f, plain)


def test_skewed_prefix_fused_equals_plain(fge):
    inp = moe_inputs("large", seed=0)
    t = 2048
    counts = np.bincount(oracle.topk_gate(inp.logits[:t], inp.k)[0].ravel(), minlength=inp.E)
    assert counts.max() > 10 * counts.mean() and (counts == 0).any()
    plain, fused = _both(fge, inp.logits[:t], inp.x_bits[:t], inp,
                         _banks(fge, inp, fge.W4_SUBNORMAL), fge.W4_SUBNORMAL)
    assert np.array_equal(fused[0], plain)
    rows = np.sort(np.random.default_rng(2).choice(t, size=48, replace=False))
    ref, _ = oracle.moe_layer_forward(inp.logits[rows], inp.x[rows], inp.k, inp.w_gu, inp.s_gu,
                                      inp.w_dn, inp.s_dn, inp.I, out_dtype="bf16")
    assert cosine(fused[0][rows], ref) >= 0.9999


def test_fused_combine_refuses_f32_output(fge):
    inp = moe_inputs("tiny", seed=1)
    banks = _banks(fge, inp, fge.W4_SUBNORMAL)
    with pytest.raises(fge.FgeError):
        fge.moe_layer_forward(to_dev(inp.logits), bf16_dev(inp.x_bits), inp.k, inp.I, *banks,
                              out_dtype=torch.float32, fused_combine=True)
