"""ctypes binding of the single-threaded C++ oracle (``oracle_ref.cpp``).

Test infrastructure only, like the rest of this package: the tests, the smoke check and
the benchmark's CPU-baseline and reference legs call it; the product library never does.
``build()`` compiles the shared object in-tree with g++ (no CUDA, no shared code with the
library); the functions below marshal numpy arrays to the C entry points and return numpy
arrays.  Each C function cites the passage it restates.
"""

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle_ref.cpp")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "liboracle_ref.so")
# -ffp-contract=off: every float64 product and sum is rounded on its own, in source order
CXXFLAGS = ["-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC"]

_lib = None


def build():
    """Compile liboracle_ref.so if the source is newer than it; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    if os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = "%s.%d.tmp" % (LIB, os.getpid())  # concurrent builds each write their own file
    r = subprocess.run([os.environ.get("CXX", "g++")] + CXXFLAGS + [SRC, "-o", tmp],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB)
    return LIB


def _p(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        i64, i32, f32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_double
        P = ctypes.POINTER
        u8p, u16p, i32p = P(ctypes.c_uint8), P(ctypes.c_uint16), P(ctypes.c_int32)
        f32p, f64p = P(ctypes.c_float), P(ctypes.c_double)
        sig = {
            "fo_e4m3_decode": (f64, [ctypes.c_uint8]),
            "fo_e4m3_encode": (ctypes.c_uint8, [f32]),
            "fo_e4m3_encode_n": (None, [f32p, i64, u8p]),
            "fo_bf16_round_n": (None, [f64p, i64, u16p]),
            "fo_e4m3_encode_selfcheck": (i64, [i32, i32]),
            "fo_quant_g128": (None, [f32p, i64, i64, u8p, f32p]),
            "fo_quant_per_tensor": (None, [f32p, i64, i64, u8p, f32p]),
            "fo_quant_per_row": (None, [f32p, i64, i64, u8p, f32p]),
            "fo_topk_gate": (None, [f32p, i64, i32, i32, i32p, f32p]),
            "fo_moe_permute": (None, [i32p, i64, i32, i32, u8p, f32p, i64, i32p, i32p, i32p,
                                      i32p, u8p, f32p]),
            "fo_grouped_gemm_w4a8": (None, [u8p, f32p, i32p, i32, u8p, f32p, i64, i64, i64,
                                            f64p]),
            "fo_swiglu_requant": (None, [f64p, i64, i64, u8p, f32p, f32p]),
            "fo_moe_combine": (None, [f32p, i32p, f32p, i64, i32, i64, f64p]),
            "fo_linear_w8a8_gemm": (None, [u8p, f32p, f32, u8p, f32, i64, i64, i64, f64p]),
            "fo_moe_layer_forward": (i32, [f32p, f32p, i64, i64, i32, i32, i64, u8p, f32p, u8p,
                                           f32p, i32, f32p]),
            "fo_mx_quant_e2m1": (None, [f32p, i64, i64, u8p, u8p]),
            "fo_grouped_gemm_mxf4_w4": (None, [u8p, u8p, i32p, i32, u8p, f32p, i64, i64, i64,
                                               f64p]),
            "fo_rmsnorm": (None, [f32p, i64, i64, f32p]),
            "fo_router_logits": (None, [f32p, f32p, i64, i64, i32, f32p]),
            "fo_identity_attention": (None, [f32p, i64, i32, i32, f32p]),
            "fo_linear_w8a8": (None, [f32p, i64, i64, u8p, f32, i64, i32, f32p]),
            "fo_moe_layer_int4_baseline": (None, [f32p, f32p, i64, i64, i32, i32, i64, u8p,
                                                  f32p, u8p, f32p, i32, f32p]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(_lib, name)
            fn.restype = res
            fn.argtypes = args
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def e4m3_decode_table():
    L = lib()
    return np.array([L.fo_e4m3_decode(c) for c in range(256)], dtype=np.float64)


def e4m3_encode(x):
    x = _c(x, np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().fo_e4m3_encode_n(_p(x, ctypes.c_float), x.size, _p(out, ctypes.c_uint8))
    return out


def encode_selfcheck(lo, hi):
    """Mismatches of the encoder against a brute-force nearest search on every float32 of
    magnitude in [2^lo, 2^hi), both signs."""
    return int(lib().fo_e4m3_encode_selfcheck(lo, hi))


def bf16_round(v):
    v = _c(v, np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().fo_bf16_round_n(_p(v, ctypes.c_double), v.size, _p(out, ctypes.c_uint16))
    return out


def _quant(fn, x, scale_shape):
    x = _c(x, np.float32)
    m, k = x.shape
    q = np.empty((m, k), dtype=np.uint8)
    s = np.empty(scale_shape(m, k), dtype=np.float32)
    fn(_p(x, ctypes.c_float), m, k, _p(q, ctypes.c_uint8), _p(s, ctypes.c_float))
    return q, s


def quant_act_g128(x):
    return _quant(lib().fo_quant_g128, x, lambda m, k: (m, k // 128))


def quant_act_per_tensor(x):
    q, s = _quant(lib().fo_quant_per_tensor, x, lambda m, k: (1,))
    return q, np.float32(s[0])


def quant_act_per_row(x):
    return _quant(lib().fo_quant_per_row, x, lambda m, k: (m,))


def topk_gate(logits, k):
    lg = _c(logits, np.float32)
    t, e = lg.shape
    ids = np.empty((t, k), dtype=np.int32)
    gates = np.empty((t, k), dtype=np.float32)
    lib().fo_topk_gate(_p(lg, ctypes.c_float), t, e, k, _p(ids, ctypes.c_int32),
                       _p(gates, ctypes.c_float))
    return ids, gates


def moe_permute(ids, num_experts, xq, xs):
    ids = _c(ids, np.int32)
    xq = _c(xq, np.uint8)
    xs = _c(xs, np.float32)
    t, k = ids.shape
    h = xq.shape[1]
    r = t * k
    out = dict(counts=np.empty(num_experts, np.int32), offsets=np.empty(num_experts + 1, np.int32),
               row_token=np.empty(r, np.int32), token_row=np.empty((t, k), np.int32),
               aq=np.empty((r, h), np.uint8), as_=np.empty((r, h // 128), np.float32))
    i32 = ctypes.c_int32
    lib().fo_moe_permute(_p(ids, i32), t, k, num_experts, _p(xq, ctypes.c_uint8),
                         _p(xs, ctypes.c_float), h, _p(out["counts"], i32),
                         _p(out["offsets"], i32), _p(out["row_token"], i32),
                         _p(out["token_row"], i32), _p(out["aq"], ctypes.c_uint8),
                         _p(out["as_"], ctypes.c_float))
    return out


def grouped_gemm_w4a8(aq, as_, offsets, w_packed, w_scale):
    aq = _c(aq, np.uint8)
    as_ = _c(as_, np.float32)
    offsets = _c(offsets, np.int32)
    w = _c(w_packed, np.uint8)
    sw = _c(w_scale, np.float32)
    r, kdim = aq.shape
    e, n, _ = w.shape
    out = np.empty((r, n), dtype=np.float64)
    lib().fo_grouped_gemm_w4a8(_p(aq, ctypes.c_uint8), _p(as_, ctypes.c_float),
                               _p(offsets, ctypes.c_int32), e, _p(w, ctypes.c_uint8),
                               _p(sw, ctypes.c_float), n, kdim, r, _p(out, ctypes.c_double))
    return out


def swiglu_requant(c, inter):
    c = _c(c, np.float64)
    r = c.shape[0]
    hq = np.empty((r, inter), np.uint8)
    hs = np.empty((r, inter // 128), np.float32)
    h = np.empty((r, inter), np.float32)
    lib().fo_swiglu_requant(_p(c, ctypes.c_double), r, inter, _p(hq, ctypes.c_uint8),
                            _p(hs, ctypes.c_float), _p(h, ctypes.c_float))
    return hq, hs, h


def moe_combine(y, token_row, gates):
    y = _c(y, np.float32)
    token_row = _c(token_row, np.int32)
    gates = _c(gates, np.float32)
    t, k = token_row.shape
    h = y.shape[1]
    out = np.empty((t, h), np.float64)
    lib().fo_moe_combine(_p(y, ctypes.c_float), _p(token_row, ctypes.c_int32),
                         _p(gates, ctypes.c_float), t, k, h, _p(out, ctypes.c_double))
    return out


def linear_w8a8_gemm(aq, sa, wq, sw, sa_rows=None):
    aq = _c(aq, np.uint8)
    wq = _c(wq, np.uint8)
    m, kdim = aq.shape
    n = wq.shape[0]
    out = np.empty((m, n), np.float64)
    rows = None if sa_rows is None else _c(sa_rows, np.float32)
    lib().fo_linear_w8a8_gemm(_p(aq, ctypes.c_uint8),
                              None if rows is None else _p(rows, ctypes.c_float),
                              float(np.float32(sa)), _p(wq, ctypes.c_uint8),
                              float(np.float32(sw)), m, n, kdim, _p(out, ctypes.c_double))
    return out


def moe_layer_forward(logits, x_f32, k, w_gate_up, s_gate_up, w_down, s_down, inter,
                      out_dtype="bf16"):
    """The whole layer in one single-threaded C++ call; returns float32 [T, H]."""
    lg = _c(logits, np.float32)
    x = _c(x_f32, np.float32)
    wgu, sgu = _c(w_gate_up, np.uint8), _c(s_gate_up, np.float32)
    wdn, sdn = _c(w_down, np.uint8), _c(s_down, np.float32)
    t, h = x.shape
    e = wgu.shape[0]
    out = np.empty((t, h), np.float32)
    f, u = ctypes.c_float, ctypes.c_uint8
    lib().fo_moe_layer_forward(_p(lg, f), _p(x, f), t, h, e, k, inter, _p(wgu, u), _p(sgu, f),
                               _p(wdn, u), _p(sdn, f), 1 if out_dtype == "f32" else 0,
                               _p(out, f))
    return out


def mx_quant_e2m1(x):
    """MXFP4: (codes uint8 [M, K/2], element 2b in the low nibble; scales uint8 [M, K/32])."""
    x = _c(x, np.float32)
    m, k = x.shape
    packed = np.zeros((m, k // 2), np.uint8)
    scales = np.empty((m, k // 32), np.uint8)
    lib().fo_mx_quant_e2m1(_p(x, ctypes.c_float), m, k, _p(packed, ctypes.c_uint8),
                           _p(scales, ctypes.c_uint8))
    return packed, scales


def grouped_gemm_mxf4_w4(codes, scales, offsets, w_packed, w_scale):
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    offsets = _c(offsets, np.int32)
    w = _c(w_packed, np.uint8)
    sw = _c(w_scale, np.float32)
    r, kh = codes.shape
    e, n, _ = w.shape
    out = np.empty((r, n), dtype=np.float64)
    lib().fo_grouped_gemm_mxf4_w4(_p(codes, ctypes.c_uint8), _p(scales, ctypes.c_uint8),
                                  _p(offsets, ctypes.c_int32), e, _p(w, ctypes.c_uint8),
                                  _p(sw, ctypes.c_float), n, 2 * kh, r, _p(out, ctypes.c_double))
    return out


def rmsnorm(h):
    h = _c(h, np.float32)
    out = np.empty_like(h)
    lib().fo_rmsnorm(_p(h, ctypes.c_float), h.shape[0], h.shape[1], _p(out, ctypes.c_float))
    return out


def router_logits(xn, w_router):
    xn = _c(xn, np.float32)
    w = _c(w_router, np.float32)
    out = np.empty((xn.shape[0], w.shape[0]), np.float32)
    lib().fo_router_logits(_p(xn, ctypes.c_float), _p(w, ctypes.c_float), xn.shape[0],
                           xn.shape[1], w.shape[0], _p(out, ctypes.c_float))
    return out


def identity_attention(v, n_heads, n_kv_heads):
    v = _c(v, np.float32)
    out = np.empty((v.shape[0], n_heads * 128), np.float32)
    lib().fo_identity_attention(_p(v, ctypes.c_float), v.shape[0], n_heads, n_kv_heads,
                                _p(out, ctypes.c_float))
    return out


def linear_w8a8(x_f32, wq, sw, rows=False):
    """Dense projection (per-tensor or row-wise activation scales), bf16 values as float32."""
    x = _c(x_f32, np.float32)
    wq = _c(wq, np.uint8)
    out = np.empty((x.shape[0], wq.shape[0]), np.float32)
    lib().fo_linear_w8a8(_p(x, ctypes.c_float), x.shape[0], x.shape[1], _p(wq, ctypes.c_uint8),
                         float(np.float32(sw)), wq.shape[0], 1 if rows else 0,
                         _p(out, ctypes.c_float))
    return out


def moe_layer_int4_baseline(logits, x_f32, k, w_gate_up, s_gate_up, w_down, s_down, inter,
                            out_dtype="bf16"):
    """Per-token int4 expert dispatch in float64, token by token; float32 [T, H]."""
    lg = _c(logits, np.float32)
    x = _c(x_f32, np.float32)
    wgu, sgu = _c(w_gate_up, np.uint8), _c(s_gate_up, np.float32)
    wdn, sdn = _c(w_down, np.uint8), _c(s_down, np.float32)
    t, h = x.shape
    out = np.empty((t, h), np.float32)
    f, u = ctypes.c_float, ctypes.c_uint8
    lib().fo_moe_layer_int4_baseline(_p(lg, f), _p(x, f), t, h, wgu.shape[0], k, inter,
                                     _p(wgu, u), _p(sgu, f), _p(wdn, u), _p(sdn, f),
                                     1 if out_dtype == "f32" else 0, _p(out, f))
    return out


def stacked_prefill(h0, layers, k, inter, n_heads, n_kv_heads):
    """The stacked prefill layers, each step a C++ call (same layer order and readings as the
    numpy ``stacked_prefill``): xn = RMSNorm(h); v = W8A8(xn); attn = identity(v);
    h += W8A8(attn); xn2 = RMSNorm(h); logits = router(xn2); h += MoE(xn2), h in float32.
    Returns (h float32 [T, H], list of per-layer routing ids)."""
    h = np.asarray(h0, dtype=np.float32).copy()
    routes = []
    for lw in layers:
        xn = rmsnorm(h)
        v = linear_w8a8(xn, lw["wv"], lw["sv"])
        o = linear_w8a8(identity_attention(v, n_heads, n_kv_heads), lw["wo"], lw["so"])
        h = (h.astype(np.float64) + o.astype(np.float64)).astype(np.float32)
        xn2 = rmsnorm(h)
        logits = router_logits(xn2, lw["w_router"])
        routes.append(topk_gate(logits, k)[0])
        y = moe_layer_forward(logits, xn2, k, lw["w_gu"], lw["s_gu"], lw["w_dn"], lw["s_dn"],
                              inter, out_dtype="bf16")
        h = (h.astype(np.float64) + y.astype(np.float64)).astype(np.float32)
    return h, routes
