"""Dense per-tensor W8A8 projection at the full workload sizes (N=6656, K=2560,
M in {16, 256, 2048, 8192}) against the oracle: the activation codes and scale bit-exact over
the whole tensor, the GEMM on sampled rows within the GEMM rule."""

import numpy as np
import pytest

import oracle
from util import bf16_dev, check_gemm, host, to_dev
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
