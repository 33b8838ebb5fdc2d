"""fge_linear_w8a8_noalloc: the dense W8A8 projection for callers that cannot allocate device
memory (hosts that own all device memory through their own pool, latency-critical paths that
must not call cudaMalloc, foreign-language hosts without a device allocator).  Its scratch is
a fixed array inside the library, so the caller passes only x, the weights and y.

Checked through the C ABI: bit for bit against the workspace-taking fge_linear_w8a8 (the same
kernels on the same operands) and within the GEMM rule against the oracle, on two calls in a
row (the second with a much smaller input, so a scale left over from the first call would
show), with the scratch's device status word read back as 0 after each call; the largest
accepted size (exactly the scratch's capacity) and M = 0 (nothing written) are covered too.
Kept in its own file, collected last.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from util import bf16_dev, check_gemm, host, to_dev
from workloads import dense_inputs, to_bf16

pytestmark = pytest.mark.gpu

EXCEEDS_STATIC_SCRATCH = 9
SCRATCH_BYTES = 16 << 20
HEADER_BYTES = 256


def _noalloc(fge, x, wq, w_scale, y):
    m, k = x.shape
    n = wq.shape[0]
    return fge.lib().fge_linear_w8a8_noalloc(
        ctypes.c_void_p(x.data_ptr()), m, k, ctypes.c_void_p(wq.data_ptr()),
        ctypes.c_void_p(w_scale.data_ptr()), n, ctypes.c_void_p(y.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _status(fge):
    out = ctypes.c_int32(-1)
    assert fge.lib().fge_linear_w8a8_noalloc_status(
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream), ctypes.byref(out)) == 0
    return out.value


def _check_against_oracle(x_bits_dev, wq_np, sw_np, got, rows=None):
    xb = host(x_bits_dev).astype(np.float32)
    xq, sa = oracle.quant_act_per_tensor(xb)
    sel = slice(None) if rows is None else rows
    ref = oracle.linear_w8a8_gemm(xq[sel], sa, wq_np, sw_np)
    absref = (float(sa) * float(sw_np)) * (np.abs(oracle.e4m3_decode(xq[sel]))
                                           @ np.abs(oracle.e4m3_decode(wq_np)).T)
    check_gemm(got[sel], ref, absref, True)


@pytest.mark.parametrize("m", [1, 16, 300])
def test_noalloc_matches_workspace_entry_point_and_oracle_on_two_calls(fge, m):
    d = dense_inputs(m)
    wq_np, sw_np = oracle.quant_act_per_tensor(d.w)
    wq = to_dev(wq_np)
    sw = to_dev(np.array([sw_np], np.float32))
    x1 = bf16_dev(d.x_bits)
    # second input: other rows, 1000x smaller, so the first call's amax would be wrong here
    rng = np.random.default_rng(99 + m)
    x2 = bf16_dev(to_bf16(rng.standard_normal((m, d.K)).astype(np.float32) * 1e-3)[0])
    for x in (x1, x2):
        y_new = torch.full((x.shape[0], d.N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _noalloc(fge, x, wq, sw, y_new) == 0
        assert _status(fge) == 0
        y_ref = fge.linear_w8a8(x, wq, sw)
        torch.cuda.synchronize()
        got = host(y_new).astype(np.float64)
        assert np.all(np.isfinite(got))
        assert np.array_equal(got, host(y_ref).astype(np.float64))
        _check_against_oracle(x, wq_np, sw_np, got)


def test_noalloc_accepts_exactly_its_capacity(fge):
    k, n = 256, 256
    m = (SCRATCH_BYTES - HEADER_BYTES) // k     # M*K == the scratch's activation capacity
    assert m * k == SCRATCH_BYTES - HEADER_BYTES
    rng = np.random.default_rng(7)
    bits, _ = to_bf16(rng.standard_normal((m, k)).astype(np.float32))
    x = bf16_dev(bits)
    wq_np, sw_np = oracle.quant_act_per_tensor((rng.standard_normal((n, k)) * 0.02).astype(np.float32))
    wq = to_dev(wq_np)
    sw = to_dev(np.array([sw_np], np.float32))
    y = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(fge, x, wq, sw, y) == 0
    assert _status(fge) == 0
    y_ref = fge.linear_w8a8(x, wq, sw)
    torch.cuda.synchronize()
    got = host(y).astype(np.float64)
    assert np.array_equal(got, host(y_ref).astype(np.float64))
    rows = np.sort(rng.choice(m, size=256, replace=False))
    _check_against_oracle(x, wq_np, sw_np, got, rows)


def test_noalloc_empty_input_writes_nothing(fge):
    k, n = 2560, 256
    x = torch.zeros((4, k), dtype=torch.bfloat16, device="cuda")[:0]  # a valid, empty view
    wq = torch.zeros((n, k), dtype=torch.uint8, device="cuda")
    sw = torch.ones(1, dtype=torch.float32, device="cuda")
    sentinel = torch.full((4, n), 3.0, dtype=torch.bfloat16, device="cuda")
    y = sentinel[:0]
    assert _noalloc(fge, x, wq, sw, y) == 0
    torch.cuda.synchronize()
    assert torch.all(sentinel == 3.0)


def test_noalloc_rejects_sizes_beyond_its_scratch(fge):
    k = 2560
    m = (SCRATCH_BYTES - HEADER_BYTES) // k + 1   # one row too many
    x = torch.empty((m, k), dtype=torch.bfloat16, device="cuda")
    wq = torch.empty((256, k), dtype=torch.uint8, device="cuda")
    sw = torch.ones(1, dtype=torch.float32, device="cuda")
    y = torch.empty((m, 256), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(fge, x, wq, sw, y) == EXCEEDS_STATIC_SCRATCH
    assert "scratch" in fge.status_string(EXCEEDS_STATIC_SCRATCH)
