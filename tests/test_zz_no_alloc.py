"""fge_linear_w8a8_noalloc: the dense W8A8 projection for callers that cannot allocate device
memory (hosts that own all device memory through their own pool, latency-critical paths that
must not call cudaMalloc, foreign-language hosts without a device allocator).  Its scratch is
a fixed array inside the library, so the caller passes only x, the weights and y.

Checked through the C ABI against the workspace-taking fge_linear_w8a8 on two calls in a row
(the second with a much smaller input, so a scale left over from the first call would show),
within the GEMM tests' bf16 bound of one ulp.  Kept in its own file, collected last.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from util import bf16_dev, bf16_ulp, host, to_dev
from workloads import dense_inputs, to_bf16

pytestmark = pytest.mark.gpu

EXCEEDS_STATIC_SCRATCH = 9
SCRATCH_BYTES = 16 << 20


def _noalloc(fge, x, wq, w_scale, y):
    m, k = x.shape
    n = wq.shape[0]
    return fge.lib().fge_linear_w8a8_noalloc(
        ctypes.c_void_p(x.data_ptr()), m, k, ctypes.c_void_p(wq.data_ptr()),
        ctypes.c_void_p(w_scale.data_ptr()), n, ctypes.c_void_p(y.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_entry_point_on_two_calls(fge):
    d = dense_inputs(300)
    wq_np, sw_np = oracle.quant_act_per_tensor(d.w)
    wq = to_dev(wq_np)
    sw = to_dev(np.array([sw_np], np.float32))
    x1 = bf16_dev(d.x_bits)
    # second input: other rows, 1000x smaller, so the first call's amax would be wrong here
    rng = np.random.default_rng(99)
    x2 = bf16_dev(to_bf16(rng.standard_normal((16, d.K)).astype(np.float32) * 1e-3)[0])
    for x in (x1, x2):
        y_new = torch.full((x.shape[0], d.N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _noalloc(fge, x, wq, sw, y_new) == 0
        y_ref = fge.linear_w8a8(x, wq, sw)
        torch.cuda.synchronize()
        got, ref = host(y_new).astype(np.float64), host(y_ref).astype(np.float64)
        assert np.all(np.isfinite(got))
        assert np.all(np.abs(got - ref) <= bf16_ulp(ref))


def test_noalloc_rejects_sizes_beyond_its_scratch(fge):
    k = 2560
    m = (SCRATCH_BYTES - 256) // k + 1          # one row too many
    x = torch.empty((m, k), dtype=torch.bfloat16, device="cuda")
    wq = torch.empty((256, k), dtype=torch.uint8, device="cuda")
    sw = torch.ones(1, dtype=torch.float32, device="cuda")
    y = torch.empty((m, 256), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(fge, x, wq, sw, y) == EXCEEDS_STATIC_SCRATCH
    assert "scratch" in fge.status_string(EXCEEDS_STATIC_SCRATCH)
