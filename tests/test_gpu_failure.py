"""Failure detection without faulting the GPU: a pipeline wait that runs out reports
FGE_ERR_DEVICE_TIMEOUT through the workspace status word and the context stays usable;
bad arguments are refused on the host before anything is launched."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from util import bf16_dev, host
from workloads import to_bf16

pytestmark = pytest.mark.gpu

DEVICE_TIMEOUT, INVALID_ARG, BAD_SHAPE, MISALIGNED, WS_TOO_SMALL = 7, 1, 2, 3, 4


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _s():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def test_wait_that_never_completes_reports_timeout_and_context_survives(fge):
    ws = fge.new_workspace(256, "cuda")
    fge.clear_device_status(ws)
    assert fge.lib().fge_selftest_wait_timeout(_p(ws), 1_000_000, _s()) == 0
    assert fge.read_device_status(ws) == DEVICE_TIMEOUT
    fge.clear_device_status(ws)
    assert fge.read_device_status(ws) == 0
    # the context still runs kernels correctly afterwards
    bits, xv = to_bf16(np.random.default_rng(3).standard_normal((64, 256)).astype(np.float32))
    xq, xs = fge.fp8_quant_act(bf16_dev(bits), "g128")
    rq, rs = oracle.quant_act_g128(xv)
    assert np.array_equal(host(xq), rq) and np.array_equal(host(xs), rs)


def test_host_side_refusals(fge):
    lib = fge.lib()
    x = torch.zeros((16, 256), dtype=torch.bfloat16, device="cuda")
    xq = torch.empty((16, 256), dtype=torch.uint8, device="cuda")
    xs = torch.empty((16, 2), dtype=torch.float32, device="cuda")
    # K not a multiple of 128
    assert lib.fge_fp8_quant_act(_p(x), 16, 200, 1, _p(xq), _p(xs), None, 0, _s()) == BAD_SHAPE
    # misaligned pointer
    mis = ctypes.c_void_p(x.data_ptr() + 2)
    assert lib.fge_fp8_quant_act(mis, 16, 128, 1, _p(xq), _p(xs), None, 0, _s()) == MISALIGNED
    # per-tensor mode without a workspace
    assert lib.fge_fp8_quant_act(_p(x), 16, 256, 0, _p(xq), _p(xs), None, 0, _s()) == INVALID_ARG
    # workspace too small for the layer
    ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    lg = torch.zeros((16, 8), dtype=torch.float32, device="cuda")
    out = torch.empty((16, 256), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((8, 1024, 128), dtype=torch.uint8, device="cuda")
    sc = torch.zeros((8, 2, 1024), dtype=torch.float32, device="cuda")
    wd = torch.zeros((8, 256, 256), dtype=torch.uint8, device="cuda")
    sd = torch.zeros((8, 4, 256), dtype=torch.float32, device="cuda")
    st = lib.fge_moe_layer_forward(_p(lg), _p(x), 16, 256, 8, 2, 512, _p(w), _p(sc), _p(wd),
                                   _p(sd), 1, 0, _p(out), _p(ws), ws.numel(), _s())
    assert st == WS_TOO_SMALL
    # k > E
    st = lib.fge_moe_topk_gate(_p(lg), 16, 8, 9, _p(xq), _p(xs), _s())
    assert st == BAD_SHAPE


# ------------------------------------------------------------------ non-finite inputs
def _layer_inputs(fge):
    from workloads import moe_inputs
    inp = moe_inputs("tiny", seed=3)
    x = torch.from_numpy(inp.x_bits.view(np.int16)).view(torch.bfloat16).cuda()
    lg = torch.from_numpy(inp.logits).cuda()
    w_gu, s_gu = fge.w4_prepack(torch.from_numpy(inp.w_gu).cuda(),
                                torch.from_numpy(inp.s_gu).cuda(), True)
    w_dn, s_dn = fge.w4_prepack(torch.from_numpy(inp.w_dn).cuda(),
                                torch.from_numpy(inp.s_dn).cuda())
    ws = fge.new_workspace(fge.workspace_bytes(fge.OP_MOE_LAYER, inp.T, inp.H, inp.I, inp.E,
                                               inp.k), x.device)
    return inp, x, lg, (w_gu, s_gu, w_dn, s_dn), ws


@pytest.mark.parametrize("bad", [float("nan"), float("inf"), -float("inf")])
def test_layer_reports_a_nonfinite_activation(fge, bad):
    inp, x, lg, banks, ws = _layer_inputs(fge)
    fge.clear_device_status(ws)
    fge.moe_layer_forward(lg, x, inp.k, inp.I, *banks, workspace=ws, out_dtype=torch.float32)
    assert fge.read_device_status(ws) == 0          # finite inputs: nothing reported
    x2 = x.clone()
    x2[5, 17] = bad
    fge.moe_layer_forward(lg, x2, inp.k, inp.I, *banks, workspace=ws, out_dtype=torch.float32)
    assert fge.read_device_status(ws) == fge.ERR_NONFINITE
    fge.clear_device_status(ws)                     # and the context keeps working
    out = fge.moe_layer_forward(lg, x, inp.k, inp.I, *banks, workspace=ws,
                                out_dtype=torch.float32)
    assert fge.read_device_status(ws) == 0 and torch.isfinite(out).all()


@pytest.mark.parametrize("mode", ["tensor", "g128", "row"])
def test_quantizers_report_a_nonfinite_activation(fge, mode):
    x = torch.randn((64, 512), device="cuda").to(torch.bfloat16)
    x[3, 200] = float("inf")
    ws = fge.new_workspace(fge.workspace_bytes(fge.OP_QUANT_PER_TENSOR, 64, 512), x.device)
    fge.clear_device_status(ws)
    lib = fge.lib()
    xq = torch.empty((64, 512), dtype=torch.uint8, device="cuda")
    xs = torch.empty((64 * 4,), dtype=torch.float32, device="cuda")
    m = {"tensor": fge.SCALE_PER_TENSOR, "g128": fge.SCALE_PER_TOKEN_G128,
         "row": fge.SCALE_PER_ROW}[mode]
    st = lib.fge_fp8_quant_act(ctypes.c_void_p(x.data_ptr()), 64, 512, m,
                               ctypes.c_void_p(xq.data_ptr()), ctypes.c_void_p(xs.data_ptr()),
                               ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    assert fge.read_device_status(ws) == fge.ERR_NONFINITE


def test_ledger_counts_launches(fge):
    inp, x, lg, banks, ws = _layer_inputs(fge)
    fge.reset_ledger()
    fge.moe_layer_forward(lg, x, inp.k, inp.I, *banks, workspace=ws, out_dtype=torch.float32)
    wq = torch.zeros((256, 512), dtype=torch.uint8, device="cuda")
    sw = torch.ones(1, dtype=torch.float32, device="cuda")
    fge.linear_w8a8(torch.randn((16, 512), device="cuda").to(torch.bfloat16), wq, sw)
    fge.linear_w8a8(torch.randn((300, 512), device="cuda").to(torch.bfloat16), wq, sw)
    torch.cuda.synchronize()
    led = fge.ledger()
    assert led["layers"] == 1 and led["grouped_gemms"] == 2
    assert led["dense_decode_tile"] == 1 and led["dense_row_tile"] == 1
    assert led["refused"] == 0 and led["calls"] >= 3
