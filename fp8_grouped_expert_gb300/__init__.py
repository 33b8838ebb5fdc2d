"""Thin Python binding of libfge (include/fge.h): W4A8 grouped-expert MoE prefill and dense
per-tensor W8A8 projections on one GB300 (sm_103a).

Argument marshalling only: every step runs in the library's CUDA kernels.  PyTorch supplies
device memory (including workspaces, allocated here on the caller's behalf) and the
current stream.  There is no fallback: if libfge.so is missing or the device is not
sm_103, calls raise.
"""

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfge.so")

# enums of include/fge.h
OK = 0
ERR_DEVICE_TIMEOUT, ERR_NONFINITE = 7, 10
SCALE_PER_TENSOR, SCALE_PER_TOKEN_G128, SCALE_PER_ROW = 0, 1, 2
DTYPE_BF16, DTYPE_F32 = 0, 1
EPI_STORE, EPI_SWIGLU_REQUANT = 0, 1
W4_LUT, W4_SUBNORMAL = 0, 1
OP_QUANT_PER_TENSOR, OP_PERMUTE, OP_GROUPED_GEMM, OP_LINEAR_W8A8, OP_MOE_LAYER = range(5)
OP_DISPATCH_BASELINE = 5
OP_LINEAR_W8A8_ROWS = 6

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int
_SZ = ctypes.c_size_t

# name -> argtypes (restype is int status unless listed in _RESTYPES)
SIGNATURES = {
    "fge_version": [],
    "fge_init": [_I],
    "fge_status_string": [_I],
    "fge_workspace_bytes": [_I, _I64, _I64, _I64, _I, _I],
    "fge_clear_device_status": [_P, _P],
    "fge_read_ledger": [_P],
    "fge_reset_ledger": [],
    "fge_read_device_status": [_P, _P, ctypes.POINTER(ctypes.c_int32)],
    "fge_fp8_quant_act": [_P, _I64, _I64, _I, _P, _P, _P, _SZ, _P],
    "fge_mx_quant_e2m1": [_P, _I64, _I64, _P, _P, _P],
    "fge_moe_topk_gate": [_P, _I64, _I, _I, _P, _P, _P],
    "fge_moe_permute": [_P, _I64, _I, _I, _P, _P, _I64, _P, _P, _P, _P, _P, _P, _SZ, _P],
    "fge_moe_permute_quant": [_P, _I64, _I, _I, _P, _I64, _P, _P, _P, _P, _P, _P, _SZ, _P],
    "fge_w4_prepack": [_P, _P, _I, _I64, _I64, _I, _I, _P, _P, _P],
    "fge_grouped_gemm_w4a8": [_P, _P, _P, _I64, _P, _P, _I, _I64, _I64, _I, _I, _I, _P, _P, _P,
                              _SZ, _P],
    "fge_grouped_gemm_mxf4_w4": [_P, _P, _P, _I64, _P, _P, _I, _I64, _I64, _I, _I, _P, _P, _SZ,
                                 _P],
    "fge_grouped_gemm_w4a8_gather": [_P, _P, _I64, _P, _P, _I64, _P, _P, _I, _I64, _I64, _I,
                                     _I, _I, _P, _P, _P, _SZ, _P],
    "fge_swiglu_quant": [_P, _I64, _I64, _P, _P, _P],
    "fge_moe_combine": [_P, _I, _P, _P, _I64, _I, _I64, _I, _P, _P],
    "fge_moe_combine_staged": [_P, _P, _P, _I64, _I, _I64, _I, _P, _P, _SZ, _P],
    "fge_gemm_w8a8": [_P, _P, _I64, _I64, _P, _P, _I64, _I, _P, _P, _SZ, _P],
    "fge_linear_w8a8": [_P, _I64, _I64, _P, _P, _I64, _P, _P, _SZ, _P],
    "fge_gemm_w8a8_rows": [_P, _P, _I64, _I64, _P, _P, _I64, _I, _P, _P, _SZ, _P],
    "fge_linear_w8a8_rows": [_P, _I64, _I64, _P, _P, _I64, _P, _P, _SZ, _P],
    "fge_moe_layer_per_token_dispatch": [_P, _P, _I64, _I64, _I, _I, _I64, _P, _P, _P, _P, _I,
                                         _P, _P, _SZ, _P],
    "fge_linear_w8a8_noalloc": [_P, _I64, _I64, _P, _P, _I64, _P, _P],
    "fge_linear_w8a8_noalloc_status": [_P, ctypes.POINTER(ctypes.c_int32)],
    "fge_moe_layer_forward": [_P, _P, _I64, _I64, _I, _I, _I64, _P, _P, _P, _P, _I, _I, _P, _P,
                              _SZ, _P],
    "fge_moe_layer_forward_fused_combine": [_P, _P, _I64, _I64, _I, _I, _I64, _P, _P, _P, _P,
                                            _I, _P, _P, _SZ, _P],
    "fge_selftest_wait_timeout": [_P, _I64, _P],
    "fge_rmsnorm": [_P, _I64, _I64, ctypes.c_float, _P, _P],
    "fge_router_logits": [_P, _P, _I64, _I64, _I, _P, _P],
    "fge_identity_attention": [_P, _I64, _I, _I, _P, _P],
    "fge_residual_add": [_P, _P, _I, _I64, _P],
    "fge_residual_rmsnorm": [_P, _P, _I, _I64, _I64, ctypes.c_float, _P, _P],
}
_RESTYPES = {"fge_version": ctypes.c_int, "fge_status_string": ctypes.c_char_p,
             "fge_workspace_bytes": ctypes.c_size_t}

_lib = None
_inited = set()


class FgeError(RuntimeError):
    pass


def lib():
    """The loaded libfge (ctypes).  Raises if the in-tree library has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise FgeError("libfge.so is not built (run fp8_grouped_expert_gb300.build.build())")
        handle = ctypes.CDLL(LIB_PATH)
        for name, args in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.argtypes = args
            fn.restype = _RESTYPES.get(name, ctypes.c_int)
        _lib = handle
    return _lib


def status_string(code):
    return lib().fge_status_string(code).decode()


def _check(code, what):
    if code != OK:
        raise FgeError("%s failed: %s (%d)" % (what, status_string(code), code))


def _ensure_init(device):
    idx = device.index if device.index is not None else torch.cuda.current_device()
    if idx not in _inited:
        _check(lib().fge_init(idx), "fge_init(%d)" % idx)
        _inited.add(idx)


def _stream(t):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _need(t, dtype, name):
    if not t.is_cuda:
        raise FgeError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise FgeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise FgeError("%s must be contiguous" % name)


def workspace_bytes(op, a=0, b=0, c=0, E=0, k=0):
    return int(lib().fge_workspace_bytes(op, a, b, c, E, k))


def new_workspace(nbytes, device):
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


class Ledger(ctypes.Structure):
    """fge_ledger (include/fge.h): host counters of this process's library calls."""
    _fields_ = [(n, ctypes.c_uint64) for n in ("calls", "refused", "layers", "grouped_gemms",
                                               "dense_decode_tile", "dense_row_tile")]


def ledger():
    """The library's call ledger as a dict."""
    led = Ledger()
    _check(lib().fge_read_ledger(ctypes.byref(led)), "fge_read_ledger")
    return {name: getattr(led, name) for name, _ in Ledger._fields_}


def reset_ledger():
    _check(lib().fge_reset_ledger(), "fge_reset_ledger")


def read_device_status(ws):
    out = ctypes.c_int32(0)
    _check(lib().fge_read_device_status(_ptr(ws), _stream(ws), ctypes.byref(out)),
           "fge_read_device_status")
    return out.value


def clear_device_status(ws):
    _check(lib().fge_clear_device_status(_ptr(ws), _stream(ws)), "fge_clear_device_status")


# ------------------------------------------------------------------------------ ops
def fp8_quant_act(x, mode="g128", workspace=None, out=None):
    """x: bf16 [M, K] -> (xq uint8 [M, K], xs float32 [M, K/128] ("g128"), [M] ("row") or
    [1] ("tensor")).  out: an (xq, xs) pair of those shapes to write into."""
    _need(x, torch.bfloat16, "x")
    _ensure_init(x.device)
    m, k = x.shape
    n_scales = {"g128": (m, k // 128), "row": (m,)}.get(mode, (1,))
    if out is not None:
        xq, xs = out
        _need(xq, torch.uint8, "xq")
        _need(xs, torch.float32, "xs")
        if tuple(xq.shape) != (m, k) or tuple(xs.shape) != n_scales:
            raise ValueError("out shapes must be %s and %s" % ((m, k), n_scales))
    else:
        xq = torch.empty((m, k), dtype=torch.uint8, device=x.device)
        xs = torch.empty(n_scales, dtype=torch.float32, device=x.device)
    if mode == "g128":
        code = lib().fge_fp8_quant_act(_ptr(x), m, k, SCALE_PER_TOKEN_G128, _ptr(xq), _ptr(xs),
                                       None, 0, _stream(x))
    elif mode == "row":
        code = lib().fge_fp8_quant_act(_ptr(x), m, k, SCALE_PER_ROW, _ptr(xq), _ptr(xs),
                                       None, 0, _stream(x))
    else:
        ws = workspace if workspace is not None else new_workspace(
            workspace_bytes(OP_QUANT_PER_TENSOR, m, k), x.device)
        code = lib().fge_fp8_quant_act(_ptr(x), m, k, SCALE_PER_TENSOR, _ptr(xq), _ptr(xs),
                                       _ptr(ws), ws.numel(), _stream(x))
    _check(code, "fge_fp8_quant_act")
    return xq, xs


def mx_quant_e2m1(x):
    """x: bf16 [M, K] (K % 32 == 0) -> (xq uint8 [M, K/2] E2M1 code pairs, low nibble first;
    xs uint8 [M, K/32] E8M0 block scale codes)."""
    _need(x, torch.bfloat16, "x")
    _ensure_init(x.device)
    m, k = x.shape
    xq = torch.empty((m, k // 2), dtype=torch.uint8, device=x.device)
    xs = torch.empty((m, k // 32), dtype=torch.uint8, device=x.device)
    _check(lib().fge_mx_quant_e2m1(_ptr(x), m, k, _ptr(xq), _ptr(xs), _stream(x)),
           "fge_mx_quant_e2m1")
    return xq, xs


def moe_topk_gate(logits, k):
    _need(logits, torch.float32, "logits")
    _ensure_init(logits.device)
    t, e = logits.shape
    ids = torch.empty((t, k), dtype=torch.int32, device=logits.device)
    gates = torch.empty((t, k), dtype=torch.float32, device=logits.device)
    _check(lib().fge_moe_topk_gate(_ptr(logits), t, e, k, _ptr(ids), _ptr(gates),
                                   _stream(logits)), "fge_moe_topk_gate")
    return ids, gates


def moe_permute(ids, num_experts, xq, xs, index_only=False):
    """Expert-contiguous routed rows.  index_only: offsets, row_token and token_row only (no
    row copy; xq/xs give the sizes), for grouped_gemm_w4a8_gather."""
    _need(ids, torch.int32, "ids")
    _need(xq, torch.uint8, "xq")
    _need(xs, torch.float32, "xs")
    _ensure_init(ids.device)
    t, k = ids.shape
    h = xq.shape[1]
    dev = ids.device
    r = t * k
    out = dict(
        offsets=torch.empty(num_experts + 1, dtype=torch.int32, device=dev),
        row_token=torch.empty(r, dtype=torch.int32, device=dev),
        token_row=torch.empty((t, k), dtype=torch.int32, device=dev),
    )
    if not index_only:
        out["aq"] = torch.empty((r, h), dtype=torch.uint8, device=dev)
        out["as_"] = torch.empty((r, h // 128), dtype=torch.float32, device=dev)
    ws = new_workspace(workspace_bytes(OP_PERMUTE, t, h, 0, num_experts, k), dev)
    _check(lib().fge_moe_permute(_ptr(ids), t, k, num_experts, _ptr(xq), _ptr(xs), h,
                                 _ptr(out["offsets"]), _ptr(out["row_token"]),
                                 _ptr(out["token_row"]), _ptr(out.get("aq")),
                                 _ptr(out.get("as_")), _ptr(ws), ws.numel(), _stream(ids)),
           "fge_moe_permute")
    return out


def moe_permute_quant(ids, num_experts, x):
    """G128 quantization folded into the permutation's row copy: x bf16 [T, H] -> the same dict
    as moe_permute (offsets, row_token, token_row, aq, as_)."""
    _need(ids, torch.int32, "ids")
    _need(x, torch.bfloat16, "x")
    _ensure_init(ids.device)
    t, k = ids.shape
    h = x.shape[1]
    dev = ids.device
    r = t * k
    out = dict(
        offsets=torch.empty(num_experts + 1, dtype=torch.int32, device=dev),
        row_token=torch.empty(r, dtype=torch.int32, device=dev),
        token_row=torch.empty((t, k), dtype=torch.int32, device=dev),
        aq=torch.empty((r, h), dtype=torch.uint8, device=dev),
        as_=torch.empty((r, h // 128), dtype=torch.float32, device=dev),
    )
    ws = new_workspace(workspace_bytes(OP_PERMUTE, t, h, 0, num_experts, k), dev)
    _check(lib().fge_moe_permute_quant(_ptr(ids), t, k, num_experts, _ptr(x), h,
                                       _ptr(out["offsets"]), _ptr(out["row_token"]),
                                       _ptr(out["token_row"]), _ptr(out["aq"]), _ptr(out["as_"]),
                                       _ptr(ws), ws.numel(), _stream(ids)), "fge_moe_permute_quant")
    return out


def w4_prepack(w_packed, w_scale, gate_up_interleave=False, fmt=W4_SUBNORMAL):
    """Canonical bank uint8 [E, N, K/2] + scales [E, N, K/128] -> kernel layout
    (uint8 [E, N, K/2], float32 [E, K/128, N])."""
    _need(w_packed, torch.uint8, "w_packed")
    _need(w_scale, torch.float32, "w_scale")
    _ensure_init(w_packed.device)
    e, n, kh = w_packed.shape
    k = kh * 2
    wd = torch.empty_like(w_packed)
    sd = torch.empty((e, k // 128, n), dtype=torch.float32, device=w_packed.device)
    _check(lib().fge_w4_prepack(_ptr(w_packed), _ptr(w_scale), e, n, k,
                                1 if gate_up_interleave else 0, fmt, _ptr(wd), _ptr(sd),
                                _stream(w_packed)), "fge_w4_prepack")
    return wd, sd


def grouped_gemm_w4a8(aq, as_, offsets, w_dev, s_dev, fmt=W4_SUBNORMAL, epilogue="store",
                      out_dtype=torch.float32, workspace=None, out=None, scales=None):
    """Grouped W4A8 GEMM; epilogue 'store' -> out [R, N]; 'swiglu' -> (hq [R, N/2], hs).

    out (and, for 'swiglu', scales) may be passed preallocated; rows past offsets[E] are
    then left as they were.  Otherwise they are allocated zero-filled."""
    _need(aq, torch.uint8, "aq")
    _need(as_, torch.float32, "as_")
    _need(offsets, torch.int32, "offsets")
    _ensure_init(aq.device)
    r, k = aq.shape
    e, n, _ = w_dev.shape
    dev = aq.device
    ws = workspace if workspace is not None else new_workspace(
        workspace_bytes(OP_GROUPED_GEMM), dev)
    if epilogue == "swiglu":
        if out is None:
            out = torch.zeros((r, n // 2), dtype=torch.uint8, device=dev)
        if scales is None:
            scales = torch.zeros((r, n // 256), dtype=torch.float32, device=dev)
        _need(out, torch.uint8, "out")
        _need(scales, torch.float32, "scales")
        if tuple(out.shape) != (r, n // 2) or tuple(scales.shape) != (r, n // 256):
            raise FgeError("out/scales must be [R, N/2] / [R, N/256]")
        epi, od = EPI_SWIGLU_REQUANT, DTYPE_BF16
    else:
        if out is None:
            out = torch.zeros((r, n), dtype=out_dtype, device=dev)
        _need(out, out_dtype, "out")
        if tuple(out.shape) != (r, n):
            raise FgeError("out must be [R, N]")
        scales = None
        epi = EPI_STORE
        od = DTYPE_F32 if out_dtype == torch.float32 else DTYPE_BF16
    _check(lib().fge_grouped_gemm_w4a8(_ptr(aq), _ptr(as_), _ptr(offsets), r, _ptr(w_dev),
                                       _ptr(s_dev), e, n, k, fmt, epi, od, _ptr(out),
                                       _ptr(scales), _ptr(ws), ws.numel(), _stream(aq)),
           "fge_grouped_gemm_w4a8")
    return (out, scales) if epilogue == "swiglu" else out


def grouped_gemm_mxf4_w4(codes, scales, offsets, w_dev, s_dev, out_dtype=torch.float32,
                         workspace=None, out=None):
    """Grouped GEMM with MXFP4 activations (codes uint8 [R, K/2], scales uint8 [R, K/32], as
    mx_quant_e2m1 returns them) and a subnormal-format int4 bank: out [R, N]."""
    _need(codes, torch.uint8, "codes")
    _need(scales, torch.uint8, "scales")
    _need(offsets, torch.int32, "offsets")
    _ensure_init(codes.device)
    r, kh = codes.shape
    k = 2 * kh
    e, n, _ = w_dev.shape
    dev = codes.device
    ws = workspace if workspace is not None else new_workspace(
        workspace_bytes(OP_GROUPED_GEMM), dev)
    if out is None:
        out = torch.zeros((r, n), dtype=out_dtype, device=dev)
    _need(out, out_dtype, "out")
    if tuple(out.shape) != (r, n) or tuple(scales.shape) != (r, k // 32):
        raise FgeError("out must be [R, N] and scales [R, K/32]")
    _check(lib().fge_grouped_gemm_mxf4_w4(_ptr(codes), _ptr(scales), _ptr(offsets), r,
                                          _ptr(w_dev), _ptr(s_dev), e, n, k, W4_SUBNORMAL,
                                          DTYPE_F32 if out_dtype == torch.float32 else DTYPE_BF16,
                                          _ptr(out), _ptr(ws), ws.numel(), _stream(codes)),
           "fge_grouped_gemm_mxf4_w4")
    return out


def grouped_gemm_w4a8_gather(xq, xs, row_token, offsets, w_dev, s_dev, fmt=W4_SUBNORMAL,
                             epilogue="store", out_dtype=torch.float32, workspace=None):
    """grouped_gemm_w4a8 with the A rows gathered from token-ordered xq [T, K] / xs [T, K/128]
    by row_token [R] (TMA row gathers in the GEMM; no permuted copy)."""
    _need(xq, torch.uint8, "xq")
    _need(xs, torch.float32, "xs")
    _need(row_token, torch.int32, "row_token")
    _need(offsets, torch.int32, "offsets")
    _ensure_init(xq.device)
    t, k = xq.shape
    r = row_token.shape[0]
    e, n, _ = w_dev.shape
    dev = xq.device
    ws = workspace if workspace is not None else new_workspace(
        workspace_bytes(OP_GROUPED_GEMM), dev)
    if epilogue == "swiglu":
        out = torch.zeros((r, n // 2), dtype=torch.uint8, device=dev)
        scales = torch.zeros((r, n // 256), dtype=torch.float32, device=dev)
        epi, od = EPI_SWIGLU_REQUANT, DTYPE_BF16
    else:
        out = torch.zeros((r, n), dtype=out_dtype, device=dev)
        scales = None
        epi = EPI_STORE
        od = DTYPE_F32 if out_dtype == torch.float32 else DTYPE_BF16
    _check(lib().fge_grouped_gemm_w4a8_gather(_ptr(xq), _ptr(xs), t, _ptr(row_token),
                                              _ptr(offsets), r, _ptr(w_dev), _ptr(s_dev), e, n,
                                              k, fmt, epi, od, _ptr(out), _ptr(scales), _ptr(ws),
                                              ws.numel(), _stream(xq)),
           "fge_grouped_gemm_w4a8_gather")
    return (out, scales) if epilogue == "swiglu" else out


def swiglu_quant(c, inter):
    _need(c, torch.float32, "c")
    _ensure_init(c.device)
    r = c.shape[0]
    hq = torch.empty((r, inter), dtype=torch.uint8, device=c.device)
    hs = torch.empty((r, inter // 128), dtype=torch.float32, device=c.device)
    _check(lib().fge_swiglu_quant(_ptr(c), r, inter, _ptr(hq), _ptr(hs), _stream(c)),
           "fge_swiglu_quant")
    return hq, hs


def moe_combine(y, token_row, gates, out_dtype=torch.bfloat16, workspace=None):
    """out[t] = sum_j gates[t, j] * y[token_row[t, j]].  With a workspace (>= 256 bytes),
    bf16 y, k <= 8 and H % 2048 == 0: fge_moe_combine_staged, the layer's own combine."""
    _need(token_row, torch.int32, "token_row")
    _need(gates, torch.float32, "gates")
    _ensure_init(y.device)
    t, k = token_row.shape
    h = y.shape[1]
    out = torch.empty((t, h), dtype=out_dtype, device=y.device)
    if workspace is not None:
        _need(y, torch.bfloat16, "y")
        _check(lib().fge_moe_combine_staged(
            _ptr(y), _ptr(token_row), _ptr(gates), t, k, h,
            DTYPE_F32 if out_dtype == torch.float32 else DTYPE_BF16, _ptr(out), _ptr(workspace),
            workspace.numel(), _stream(y)), "fge_moe_combine_staged")
        return out
    _check(lib().fge_moe_combine(_ptr(y), DTYPE_F32 if y.dtype == torch.float32 else DTYPE_BF16,
                                 _ptr(token_row), _ptr(gates), t, k, h,
                                 DTYPE_F32 if out_dtype == torch.float32 else DTYPE_BF16,
                                 _ptr(out), _stream(y)), "fge_moe_combine")
    return out


def gemm_w8a8(aq, sa, wq, sw, out_dtype=torch.bfloat16, workspace=None, out=None):
    _need(aq, torch.uint8, "aq")
    _need(wq, torch.uint8, "wq")
    _ensure_init(aq.device)
    m, k = aq.shape
    n = wq.shape[0]
    ws = workspace if workspace is not None else new_workspace(
        workspace_bytes(OP_GROUPED_GEMM), aq.device)
    if out is not None:
        _need(out, out_dtype, "out")
        if tuple(out.shape) != (m, n):
            raise ValueError("out must be [%d, %d]" % (m, n))
    y = out if out is not None else torch.empty((m, n), dtype=out_dtype, device=aq.device)
    _check(lib().fge_gemm_w8a8(_ptr(aq), _ptr(sa), m, k, _ptr(wq), _ptr(sw), n,
                               DTYPE_F32 if out_dtype == torch.float32 else DTYPE_BF16, _ptr(y),
                               _ptr(ws), ws.numel(), _stream(aq)), "fge_gemm_w8a8")
    return y


def linear_w8a8(x, wq, w_scale, workspace=None, out=None):
    _need(x, torch.bfloat16, "x")
    _need(wq, torch.uint8, "wq")
    _ensure_init(x.device)
    m, k = x.shape
    n = wq.shape[0]
    ws = workspace if workspace is not None else new_workspace(
        workspace_bytes(OP_LINEAR_W8A8, m, k, n), x.device)
    y = out if out is not None else torch.empty((m, n), dtype=torch.bfloat16, device=x.device)
    _check(lib().fge_linear_w8a8(_ptr(x), m, k, _ptr(wq), _ptr(w_scale), n, _ptr(y), _ptr(ws),
                                 ws.numel(), _stream(x)), "fge_linear_w8a8")
    return y


def gemm_w8a8_rows(aq, sa_rows, wq, sw, out_dtype=torch.bfloat16, workspace=None):
    """One-group W8A8 GEMM with one activation scale per row: sa_rows float32 [M]."""
    _need(aq, torch.uint8, "aq")
    _need(wq, torch.uint8, "wq")
    _need(sa_rows, torch.float32, "sa_rows")
    _ensure_init(aq.device)
    m, k = aq.shape
    n = wq.shape[0]
    ws = workspace if workspace is not None else new_workspace(
        workspace_bytes(OP_GROUPED_GEMM), aq.device)
    y = torch.empty((m, n), dtype=out_dtype, device=aq.device)
    _check(lib().fge_gemm_w8a8_rows(_ptr(aq), _ptr(sa_rows), m, k, _ptr(wq), _ptr(sw), n,
                                    DTYPE_F32 if out_dtype == torch.float32 else DTYPE_BF16,
                                    _ptr(y), _ptr(ws), ws.numel(), _stream(aq)),
           "fge_gemm_w8a8_rows")
    return y


def linear_w8a8_rows(x, wq, w_scale, workspace=None, out=None):
    """Dense projection with row-wise activation scales (per-row quant + GEMM), bf16 out."""
    _need(x, torch.bfloat16, "x")
    _need(wq, torch.uint8, "wq")
    _ensure_init(x.device)
    m, k = x.shape
    n = wq.shape[0]
    ws = workspace if workspace is not None else new_workspace(
        workspace_bytes(OP_LINEAR_W8A8_ROWS, m, k), x.device)
    y = out if out is not None else torch.empty((m, n), dtype=torch.bfloat16, device=x.device)
    _check(lib().fge_linear_w8a8_rows(_ptr(x), m, k, _ptr(wq), _ptr(w_scale), n, _ptr(y),
                                      _ptr(ws), ws.numel(), _stream(x)), "fge_linear_w8a8_rows")
    return y


def moe_layer_forward(logits, x, k, inter, w_gu_dev, s_gu_dev, w_dn_dev, s_dn_dev,
                      fmt=W4_SUBNORMAL, out_dtype=torch.bfloat16, workspace=None, out=None,
                      fused_combine=False):
    """One MoE FFN layer.  fused_combine: the combine runs in the down GEMM's epilogue
    (fge_moe_layer_forward_fused_combine; bf16 output, bit-identical to the plain call)."""
    _need(logits, torch.float32, "logits")
    _need(x, torch.bfloat16, "x")
    _ensure_init(x.device)
    t, h = x.shape
    e = logits.shape[1]
    if fused_combine and out_dtype != torch.bfloat16:
        raise FgeError("fused_combine writes a bf16 output")
    ws = workspace if workspace is not None else new_workspace(
        workspace_bytes(OP_MOE_LAYER, t, h, inter, e, k), x.device)
    y = out if out is not None else torch.empty((t, h), dtype=out_dtype, device=x.device)
    if fused_combine:
        _need(y, torch.bfloat16, "out")
        _check(lib().fge_moe_layer_forward_fused_combine(
            _ptr(logits), _ptr(x), t, h, e, k, inter, _ptr(w_gu_dev), _ptr(s_gu_dev),
            _ptr(w_dn_dev), _ptr(s_dn_dev), fmt, _ptr(y), _ptr(ws), ws.numel(), _stream(x)),
            "fge_moe_layer_forward_fused_combine")
        return y
    _check(lib().fge_moe_layer_forward(_ptr(logits), _ptr(x), t, h, e, k, inter, _ptr(w_gu_dev),
                                       _ptr(s_gu_dev), _ptr(w_dn_dev), _ptr(s_dn_dev), fmt,
                                       DTYPE_F32 if out_dtype == torch.float32 else DTYPE_BF16,
                                       _ptr(y), _ptr(ws), ws.numel(), _stream(x)),
           "fge_moe_layer_forward")
    return y


class HostLayerPipeline:
    """MoE layer calls from pinned host buffers to pinned host buffers, with the copies
    overlapped with the layers: step i's inputs go up on one copy stream while step i-1
    computes, and step i-1's output comes down on another while step i computes.  Two
    device buffers per input and output alternate between steps; events order the three
    streams.  Every step still moves its own inputs up and its own result down.

    submit() enqueues one step and returns at once; finish() waits for every step.  With
    graphs=True (the default) the layer call of each slot is captured once as a CUDA graph
    and replayed, so its 8 kernels launch without host gaps."""

    def __init__(self, tokens, hidden, experts, k, inter, w_gu_dev, s_gu_dev, w_dn_dev,
                 s_dn_dev, fmt=W4_SUBNORMAL, out_dtype=torch.bfloat16, device=None,
                 graphs=True):
        dev = torch.device(device if device is not None else "cuda")
        _ensure_init(dev)
        self.k, self.inter, self.fmt, self.out_dtype = k, inter, fmt, out_dtype
        self.banks = (w_gu_dev, s_gu_dev, w_dn_dev, s_dn_dev)
        self.x = [torch.empty((tokens, hidden), dtype=torch.bfloat16, device=dev)
                  for _ in range(2)]
        self.logits = [torch.empty((tokens, experts), dtype=torch.float32, device=dev)
                       for _ in range(2)]
        self.out = [torch.empty((tokens, hidden), dtype=out_dtype, device=dev) for _ in range(2)]
        self.ws = new_workspace(workspace_bytes(OP_MOE_LAYER, tokens, hidden, inter, experts, k),
                                dev)
        self.up = torch.cuda.Stream(dev)
        self.compute = torch.cuda.Stream(dev)
        self.down = torch.cuda.Stream(dev)
        ev = lambda: torch.cuda.Event()  # noqa: E731
        self.inputs_ready = [ev(), ev()]
        self.layer_done = [ev(), ev()]
        self.output_read = [ev(), ev()]
        self.used = [False, False]
        self.step = 0
        self.graphs = None
        if graphs:
            for t in self.x + self.logits:
                t.zero_()
            self._layer(0)  # first call outside capture: one-time kernel attributes
            torch.cuda.synchronize(dev)
            self.graphs = []
            for slot in range(2):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    self._layer(slot)
                self.graphs.append(g)
            torch.cuda.synchronize(dev)

    def _layer(self, slot):
        moe_layer_forward(self.logits[slot], self.x[slot], self.k, self.inter, *self.banks,
                          fmt=self.fmt, out_dtype=self.out_dtype, workspace=self.ws,
                          out=self.out[slot])

    def submit(self, x_pin, logits_pin, out_pin):
        s = self.step % 2
        if self.used[s]:  # the layer that read this slot's inputs has finished
            self.up.wait_event(self.layer_done[s])
        with torch.cuda.stream(self.up):
            self.x[s].copy_(x_pin, non_blocking=True)
            self.logits[s].copy_(logits_pin, non_blocking=True)
            self.inputs_ready[s].record(self.up)
        self.compute.wait_event(self.inputs_ready[s])
        if self.used[s]:  # this slot's previous output has been copied down
            self.compute.wait_event(self.output_read[s])
        with torch.cuda.stream(self.compute):
            if self.graphs is not None:
                self.graphs[s].replay()
            else:
                self._layer(s)
            self.layer_done[s].record(self.compute)
        self.down.wait_event(self.layer_done[s])
        with torch.cuda.stream(self.down):
            out_pin.copy_(self.out[s], non_blocking=True)
            self.output_read[s].record(self.down)
        self.used[s] = True
        self.step += 1

    def finish(self):
        for st in (self.up, self.compute, self.down):
            st.synchronize()


def moe_layer_per_token_dispatch(logits, x, k, inter, w_gu, s_gu, w_dn, s_dn,
                                 out_dtype=torch.bfloat16, workspace=None, out=None):
    """Per-token int4 dispatch baseline (canonical, unprepacked int4 banks)."""
    _need(logits, torch.float32, "logits")
    _need(x, torch.bfloat16, "x")
    _ensure_init(x.device)
    t, h = x.shape
    e = logits.shape[1]
    ws = workspace if workspace is not None else new_workspace(
        workspace_bytes(OP_DISPATCH_BASELINE, t, h, inter, e, k), x.device)
    y = out if out is not None else torch.empty((t, h), dtype=out_dtype, device=x.device)
    _check(lib().fge_moe_layer_per_token_dispatch(
        _ptr(logits), _ptr(x), t, h, e, k, inter, _ptr(w_gu), _ptr(s_gu), _ptr(w_dn), _ptr(s_dn),
        DTYPE_F32 if out_dtype == torch.float32 else DTYPE_BF16, _ptr(y), _ptr(ws), ws.numel(),
        _stream(x)), "fge_moe_layer_per_token_dispatch")
    return y


def rmsnorm(h, eps=1e-6, out=None):
    _need(h, torch.float32, "h")
    _ensure_init(h.device)
    t, d = h.shape
    y = out if out is not None else torch.empty((t, d), dtype=torch.bfloat16, device=h.device)
    _check(lib().fge_rmsnorm(_ptr(h), t, d, eps, _ptr(y), _stream(h)), "fge_rmsnorm")
    return y


def router_logits(xn, w_router, out=None):
    _need(xn, torch.bfloat16, "xn")
    _need(w_router, torch.float32, "w_router")
    _ensure_init(xn.device)
    t, d = xn.shape
    e = w_router.shape[0]
    y = out if out is not None else torch.empty((t, e), dtype=torch.float32, device=xn.device)
    _check(lib().fge_router_logits(_ptr(xn), _ptr(w_router), t, d, e, _ptr(y), _stream(xn)),
           "fge_router_logits")
    return y


def identity_attention(v, n_heads, n_kv_heads, out=None):
    _need(v, torch.bfloat16, "v")
    _ensure_init(v.device)
    t = v.shape[0]
    y = out if out is not None else torch.empty((t, n_heads * 128), dtype=torch.bfloat16,
                                                device=v.device)
    _check(lib().fge_identity_attention(_ptr(v), t, n_heads, n_kv_heads, _ptr(y), _stream(v)),
           "fge_identity_attention")
    return y


def residual_add(h, y):
    _need(h, torch.float32, "h")
    _ensure_init(h.device)
    _check(lib().fge_residual_add(_ptr(h), _ptr(y),
                                  DTYPE_F32 if y.dtype == torch.float32 else DTYPE_BF16,
                                  h.numel(), _stream(h)), "fge_residual_add")
    return h


def residual_rmsnorm(h, y, eps=1e-6, out=None):
    """h += y, then rmsnorm(h) as bf16 (the same bits as residual_add then rmsnorm)."""
    _need(h, torch.float32, "h")
    _ensure_init(h.device)
    if tuple(y.shape) != tuple(h.shape):
        raise ValueError("y must have h's shape")
    t, d = h.shape
    xn = out if out is not None else torch.empty((t, d), dtype=torch.bfloat16, device=h.device)
    _check(lib().fge_residual_rmsnorm(_ptr(h), _ptr(y),
                                      DTYPE_F32 if y.dtype == torch.float32 else DTYPE_BF16,
                                      t, d, eps, _ptr(xn), _stream(h)), "fge_residual_rmsnorm")
    return xn


# --------------------------------------------------------------------- stacked prefill
class StackedPrefill:
    """L pre-norm blocks of the stacked prefill workload, every step a C-ABI call:
    RMSNorm -> per-tensor W8A8 q/k/v (one quantization, q and k on side streams) ->
    identity attention on v -> W8A8 o -> fp32 residual
    -> RMSNorm -> fp32 router -> MoE layer (top-k, quant, permute, grouped GEMMs, combine)
    -> fp32 residual.

    layers: list of dicts with bf16 projection weights (wq_bits, wk_bits, wv_bits, wo_bits as
    uint16 numpy [rows, H], or wq, wk, wv, wo as bf16 device tensors), fp32 w_router [E, H]
    and canonical int4 banks w_gu/s_gu, w_dn/s_dn (numpy arrays or device tensors).
    Projection weights are quantized per tensor to e4m3 at load by the library's own
    quantizer; int4 banks are prepacked at load.
    """

    def __init__(self, layers, T, H, E, I, k, n_heads, n_kv_heads, device, fmt=W4_SUBNORMAL):
        import numpy as np
        self.T, self.H, self.E, self.I, self.k = T, H, E, I, k
        self.n_heads, self.n_kv = n_heads, n_kv_heads
        self.fmt = fmt
        self.dev = torch.device(device)
        _ensure_init(self.dev)
        self.layers = []
        def dev_tensor(a):
            return a.to(self.dev) if torch.is_tensor(a) else torch.from_numpy(a).to(self.dev)

        for lw in layers:
            d = {}
            for name in ("q", "k", "v", "o"):
                if "w" + name in lw:
                    wb = lw["w" + name].to(self.dev)
                else:
                    bits = np.ascontiguousarray(lw["w" + name + "_bits"]).view(np.int16)
                    wb = torch.from_numpy(bits).view(torch.bfloat16).to(self.dev)
                wq, ws = fp8_quant_act(wb, "tensor")
                d["w" + name], d["s" + name] = wq, ws
            d["w_router"] = dev_tensor(lw["w_router"])
            d["w_gu"], d["s_gu"] = w4_prepack(dev_tensor(lw["w_gu"]), dev_tensor(lw["s_gu"]),
                                              True, fmt)
            d["w_dn"], d["s_dn"] = w4_prepack(dev_tensor(lw["w_dn"]), dev_tensor(lw["s_dn"]),
                                              False, fmt)
            self.layers.append(d)
        dev = self.dev
        kv = n_kv_heads * 128
        # the o projection quantizes its own input; q, k and v share one per-tensor
        # quantization of the normed hidden state, and q and k run on side streams next to
        # the rest of the layer (the identity attention reads only v)
        self.ws_lin = new_workspace(workspace_bytes(OP_LINEAR_W8A8, T, n_heads * 128, H), dev)
        self.ws_qt = new_workspace(workspace_bytes(OP_QUANT_PER_TENSOR, T, H), dev)
        self.ws_proj = [new_workspace(workspace_bytes(OP_GROUPED_GEMM), dev) for _ in range(3)]
        self.side = [torch.cuda.Stream(dev) for _ in range(2)]
        self.xq = torch.empty((T, H), dtype=torch.uint8, device=dev)
        self.xs = torch.empty((1,), dtype=torch.float32, device=dev)
        self.ws_moe = new_workspace(workspace_bytes(OP_MOE_LAYER, T, H, I, E, k), dev)
        self.xn = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        self.q = torch.empty((T, n_heads * 128), dtype=torch.bfloat16, device=dev)
        self.kk = torch.empty((T, kv), dtype=torch.bfloat16, device=dev)
        self.v = torch.empty((T, kv), dtype=torch.bfloat16, device=dev)
        self.attn = torch.empty((T, n_heads * 128), dtype=torch.bfloat16, device=dev)
        self.o = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        self.logits = torch.empty((T, E), dtype=torch.float32, device=dev)
        self.y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)

    def forward(self, h, layers=None):
        """h: float32 [T, H] on the device, updated in place and returned.  ``layers``
        selects which layer indices to run (all, in order, by default).  Each residual add
        that a norm follows runs fused with it (fge_residual_rmsnorm, the same bits)."""
        order = list(range(len(self.layers)) if layers is None else layers)
        if not order:
            return h
        rmsnorm(h, out=self.xn)
        for n, li in enumerate(order):
            d = self.layers[li]
            main = torch.cuda.current_stream(self.dev)
            fp8_quant_act(self.xn, "tensor", workspace=self.ws_qt, out=(self.xq, self.xs))
            for side, w, sc, ws, y in zip(self.side, ("wq", "wk"), ("sq", "sk"),
                                          self.ws_proj, (self.q, self.kk)):
                side.wait_stream(main)
                with torch.cuda.stream(side):
                    gemm_w8a8(self.xq, self.xs, d[w], d[sc], workspace=ws, out=y)
            gemm_w8a8(self.xq, self.xs, d["wv"], d["sv"], workspace=self.ws_proj[2], out=self.v)
            identity_attention(self.v, self.n_heads, self.n_kv, out=self.attn)
            linear_w8a8(self.attn, d["wo"], d["so"], workspace=self.ws_lin, out=self.o)
            residual_rmsnorm(h, self.o, out=self.xn)
            router_logits(self.xn, d["w_router"], out=self.logits)
            moe_layer_forward(self.logits, self.xn, self.k, self.I, d["w_gu"], d["s_gu"],
                              d["w_dn"], d["s_dn"], fmt=self.fmt, workspace=self.ws_moe,
                              out=self.y)
            if n + 1 < len(order):
                residual_rmsnorm(h, self.y, out=self.xn)  # the next layer's first norm
            else:
                residual_add(h, self.y)
            for side in self.side:  # before the next layer rewrites xq, q and kk
                main.wait_stream(side)
        return h
