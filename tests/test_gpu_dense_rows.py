"""Dense W8A8 projection with row-wise (per-token) activation scales against the oracle:
per-row quantization bit-exact, the GEMM within the GEMM rule at the dense shapes
(N=6656, K=2560), and the error of row-wise against per-tensor scales on activations with
outlier channels (the comparison "feat(qwen4_exp) ..." section "Limits" describes)."""

import numpy as np
import pytest
import torch

import oracle
from util import bf16_dev, check_gemm, host, to_dev
from workloads import dense_activations_outlier_rows, dense_activations_outliers, dense_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("m,k", [(1, 128), (16, 2560), (257, 2560), (64, 128 * 33)])
def test_quant_per_row_bit_exact(fge, m, k):
    d = dense_inputs(m, seed=7, N=128, K=k)
    xq_g, xs_g = fge.fp8_quant_act(bf16_dev(d.x_bits), "row")
    xq, xs = oracle.quant_act_per_row(d.x)
    assert np.array_equal(host(xs_g), xs)
    assert np.array_equal(host(xq_g), xq)


def test_quant_per_row_zero_rows(fge):
    x = np.zeros((5, 256), dtype=np.float32)
    x[2, 9] = 1.5
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    xq_g, xs_g = fge.fp8_quant_act(bf16_dev(bits), "row")
    xq, xs = oracle.quant_act_per_row(x)
    assert np.array_equal(host(xs_g), xs) and np.array_equal(host(xq_g), xq)


def test_gemm_w8a8_rows_exact(fge):
    rng = np.random.default_rng(61)
    m, n, kdim = 200, 384, 512
    a = rng.integers(-8, 9, size=(m, kdim)).astype(np.float32)
    w = rng.integers(-8, 9, size=(n, kdim)).astype(np.float32)
    aq, wq = oracle.e4m3_encode(a), oracle.e4m3_encode(w)
    sa = (2.0 ** rng.integers(-6, 4, size=m)).astype(np.float32)
    sw = np.float32(2.0 ** -7)
    y = fge.gemm_w8a8_rows(to_dev(aq), to_dev(sa), to_dev(wq), to_dev(np.array([sw])),
                           out_dtype=torch.float32)
    ref = oracle.linear_w8a8_rows_gemm(aq, sa, wq, sw)
    assert np.array_equal(host(y).astype(np.float64), ref)


def _check_rows(y, xq, sa, wq, sw, rows):
    ref = oracle.linear_w8a8_rows_gemm(xq[rows], sa[rows], wq, sw)
    absref = (sa[rows].astype(np.float64)[:, None] * float(sw)) * (
        np.abs(oracle.e4m3_decode(xq[rows])) @ np.abs(oracle.e4m3_decode(wq)).T)
    check_gemm(y[rows], ref, absref, True)


@pytest.mark.parametrize("m", [1, 16, 300, 2048, 8192])
def test_linear_w8a8_rows(fge, m):
    d = dense_inputs(m, seed=8)
    wq_g, sw_g = fge.fp8_quant_act(bf16_dev(d.w_bits), "tensor")
    wq, sw = oracle.quant_act_per_tensor(d.w)
    x = bf16_dev(d.x_bits)
    xq_g, sa_g = fge.fp8_quant_act(x, "row")
    xq, sa = oracle.quant_act_per_row(d.x)
    assert np.array_equal(host(sa_g), sa) and np.array_equal(host(xq_g), xq)
    y = host(fge.linear_w8a8_rows(x, wq_g, sw_g))
    rows = np.arange(m) if m <= 300 else np.sort(
        np.random.default_rng(m).choice(m, size=48, replace=False))
    _check_rows(y, xq, sa, wq, sw, rows)


@pytest.mark.parametrize("kind", ["channels", "rows"])
def test_rowwise_vs_per_tensor_with_outliers(fge, kind):
    """Both scale schemes on the same bf16 activations (1% of channels, or 1% of rows, x20)
    and the same e4m3 weights; error against the unquantized activations times the quantized
    weights, so only the activation quantization differs.  Also times both calls."""
    m = 2048
    d = dense_inputs(16, seed=9)
    gen = dense_activations_outliers if kind == "channels" else dense_activations_outlier_rows
    xb, xf = gen(m, d.K, seed=9)
    wq_g, sw_g = fge.fp8_quant_act(bf16_dev(d.w_bits), "tensor")
    wq, sw = oracle.quant_act_per_tensor(d.w)
    x = bf16_dev(xb)
    rows = np.sort(np.random.default_rng(3).choice(m, size=64, replace=False))
    wd = oracle.e4m3_decode(wq) * float(sw)
    exact = xf[rows].astype(np.float64) @ wd.T
    results = {}
    for name, fn in (("per_tensor", fge.linear_w8a8), ("per_row", fge.linear_w8a8_rows)):
        y = host(fn(x, wq_g, sw_g))[rows]
        # mean over rows of each row's relative error: rows of ordinary size count as much
        # as the outlier rows
        results[name] = float(np.mean(np.linalg.norm(y - exact, axis=1)
                                      / np.linalg.norm(exact, axis=1)))
        for _ in range(3):
            fn(x, wq_g, sw_g)
        torch.cuda.synchronize()
        ts = []
        for _ in range(20):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn(x, wq_g, sw_g)
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        results[name + "_ms"] = float(np.median(ts))
    print("outlier %s, M=%d N=%d K=%d: mean row relative error per-tensor %.4e, per-row %.4e; "
          "time per-tensor %.4f ms, per-row %.4f ms" % (
              kind, m, d.N, d.K, results["per_tensor"], results["per_row"],
              results["per_tensor_ms"], results["per_row_ms"]))
    # e4m3 keeps 4 significant bits over a wide exponent range, so the coarser per-tensor
    # scale costs little: both schemes stay at the e4m3 error level (about 2^-5 per value,
    # averaged down over K)
    assert results["per_tensor"] < 0.05 and results["per_row"] < 0.05
    assert abs(results["per_row"] - results["per_tensor"]) < 0.1 * results["per_tensor"]
