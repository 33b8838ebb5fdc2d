"""Dense per-tensor W8A8 projection at the full workload sizes (N=6656, K=2560,
M in {16, 256, 2048, 8192}) against the oracle: the activation codes and scale bit-exact over
the whole tensor, the GEMM on sampled rows within the GEMM rule."""

import numpy as np
import pytest
import torch

import oracle
from util import DEV, bf16_dev, check_gemm, host, to_dev
from workloads import dense_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("m", [16, 256, 2048, 8192])
def test_dense_full_size(fge, m):
    d = dense_inputs(m, seed=5)
    wq_g, sw_g = fge.fp8_quant_act(bf16_dev(d.w_bits), "tensor")      # load-time quant
    wq, sw = oracle.quant_act_per_tensor(d.w)
    assert host(sw_g)[0] == sw and np.array_equal(host(wq_g), wq)
    x = bf16_dev(d.x_bits)
    xq_g, sa_g = fge.fp8_quant_act(x, "tensor")
    xq, sa = oracle.quant_act_per_tensor(d.x)
    assert host(sa_g)[0] == sa and np.array_equal(host(xq_g), xq)
    y = host(fge.linear_w8a8(x, wq_g, sw_g))
    rows = np.sort(np.random.default_rng(m).choice(m, size=min(m, 48), replace=False))
    ref = oracle.linear_w8a8_gemm(xq[rows], sa, wq, sw)
    absref = (float(sa) * float(sw)) * (np.abs(oracle.e4m3_decode(xq[rows]))
                                        @ np.abs(oracle.e4m3_decode(wq)).T)
    check_gemm(y[rows], ref, absref, True)


@pytest.mark.parametrize("m,k", [(1, 2560), (5, 2560), (16, 2560), (9, 1408), (3, 4096),
                                 (16, 4096)])
def test_decode_sizes_exact_and_repeatable(fge, m, k):
    # Decode sizes: up to K = 2560 the weight-streaming decode kernel (warp MMAs, eight warps
    # splitting K, partials added in warp order), beyond it the grouped kernel's 16-token
    # tile with K split over several CTAs per 128-feature tile.  Integer activations and
    # weights with power-of-two scales keep every partial and every sum exact, so the result
    # must equal the oracle bit for bit, and five calls must agree bit for bit.
    rng = np.random.default_rng(70 + m + k)
    n = 6656
    x = rng.integers(-8, 9, (m, k)).astype(np.float32)
    x[0, 0] = 448.0                                   # amax 448: activation scale exactly 1
    w = rng.integers(-8, 9, (n, k)).astype(np.float32)
    w[0, 0] = 448.0
    xt = torch.from_numpy(x).to(torch.bfloat16).to(DEV)
    wq_g, sw_g = fge.fp8_quant_act(torch.from_numpy(w).to(torch.bfloat16).to(DEV), "tensor")
    assert float(host(sw_g)[0]) == 1.0
    ws = fge.new_workspace(fge.workspace_bytes(fge.OP_LINEAR_W8A8, m, k, n), DEV)
    assert ws.numel() > fge.workspace_bytes(fge.OP_LINEAR_W8A8, m, k)   # room for the split
    outs = [host(fge.linear_w8a8(xt, wq_g, sw_g, workspace=ws)) for _ in range(5)]
    xq, sa = oracle.quant_act_per_tensor(x)
    wq, sw = oracle.quant_act_per_tensor(w)
    ref = oracle.linear_w8a8_gemm(xq, sa, wq, sw)
    ref_bf16 = torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16).float().numpy()
    assert np.array_equal(outs[0], ref_bf16)
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])
