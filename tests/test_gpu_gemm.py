"""GPU parity of the tcgen05 grouped GEMM (int4 bank, both bank formats) and of the same
kernel run as the dense per-tensor W8A8 GEMM, against the float64 oracle on identical
quantized operands.  Exact cases must match bit for bit; random cases meet the normwise
2e-3 / elementwise (1 bf16 ulp + 1e-5 sum|as*sw*a*w|) bound."""

import numpy as np
import pytest
import torch

import oracle
from util import abs_grouped, bf16_dev, check_gemm, host, to_dev
from workloads import dense_inputs, pack_int4

pytestmark = pytest.mark.gpu

FORMATS = ["lut", "subnormal"]


def _fmt(fge, name):
    return fge.W4_LUT if name == "lut" else fge.W4_SUBNORMAL


def _prepack(fge, wp, ws, fmt, interleave=False):
    return fge.w4_prepack(to_dev(wp), to_dev(ws), gate_up_interleave=interleave,
                          fmt=_fmt(fge, fmt))


def _routed_case(rng, t, e, k, h):
    lg = (rng.standard_normal((t, e)) - 1.1 * np.log(np.arange(1, e + 1))).astype(np.float32)
    ids, _ = oracle.topk_gate(lg, k)
    x = rng.standard_normal((t, h)).astype(np.float32)
    xq, xs = oracle.quant_act_g128(x)
    return oracle.moe_permute(ids, e, xq, xs)


@pytest.mark.parametrize("fmt", FORMATS)
def test_grouped_exact_small_integers(fge, fmt):
    # |a| <= 16 integers, scales in {1, 2} x {2^-6, 2^-5}: every partial and the fp32
    # accumulation are exact, so the kernel must reproduce the oracle bit for bit.
    rng = np.random.default_rng(21)
    counts = [130, 0, 70, 1]
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    r, n, kdim = int(offsets[-1]), 256, 384
    a = rng.integers(-16, 17, size=(r, kdim)).astype(np.float32)
    aq = oracle.e4m3_encode(a)
    as_ = rng.choice([1.0, 2.0], size=(r, 3)).astype(np.float32)
    q = rng.integers(-8, 8, size=(4, n, kdim))
    wp = pack_int4(q)
    ws = rng.choice([2.0 ** -6, 2.0 ** -5], size=(4, n, 3)).astype(np.float32)
    wd, sd = _prepack(fge, wp, ws, fmt)
    out = fge.grouped_gemm_w4a8(to_dev(aq), to_dev(as_), to_dev(offsets), wd, sd,
                                fmt=_fmt(fge, fmt), out_dtype=torch.float32)
    ref = oracle.grouped_gemm_w4a8(aq, as_, offsets, wp, ws)
    assert np.array_equal(host(out).astype(np.float64), ref)


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("t,e,k,h,n", [(64, 8, 2, 256, 1024), (97, 8, 2, 512, 256),
                                       (300, 16, 4, 1024, 384)])
def test_grouped_random(fge, fmt, out_dtype, t, e, k, h, n):
    rng = np.random.default_rng(t + n)
    p = _routed_case(rng, t, e, k, h)
    q = rng.integers(-8, 8, size=(e, n, h))
    wp = pack_int4(q)
    ws = rng.uniform(0.002, 0.02, size=(e, n, h // 128)).astype(np.float32)
    wd, sd = _prepack(fge, wp, ws, fmt)
    out = fge.grouped_gemm_w4a8(to_dev(p["aq"]), to_dev(p["as_"]), to_dev(p["offsets"]), wd, sd,
                                fmt=_fmt(fge, fmt), out_dtype=out_dtype)
    ref = oracle.grouped_gemm_w4a8(p["aq"], p["as_"], p["offsets"], wp, ws)
    absref = abs_grouped(p["aq"], p["as_"], p["offsets"], wp, ws)
    check_gemm(host(out), ref, absref, out_dtype == torch.bfloat16)


def test_grouped_mid_shape(fge):
    # gate_up of the mid layer on 512 tokens: E=64, N=1536, K=2048, top-8 (R=4096)
    rng = np.random.default_rng(31)
    p = _routed_case(rng, 512, 64, 8, 2048)
    wp = pack_int4(rng.integers(-8, 8, size=(64, 1536, 2048)))
    ws = rng.uniform(0.002, 0.02, size=(64, 1536, 16)).astype(np.float32)
    wd, sd = _prepack(fge, wp, ws, "subnormal")
    out = fge.grouped_gemm_w4a8(to_dev(p["aq"]), to_dev(p["as_"]), to_dev(p["offsets"]), wd, sd,
                                out_dtype=torch.bfloat16)
    ref = oracle.grouped_gemm_w4a8(p["aq"], p["as_"], p["offsets"], wp, ws)
    absref = abs_grouped(p["aq"], p["as_"], p["offsets"], wp, ws)
    check_gemm(host(out), ref, absref, True)


@pytest.mark.parametrize("fmt", FORMATS)
def test_swiglu_epilogue(fge, fmt):
    rng = np.random.default_rng(41)
    t, e, k, h, inter = 200, 8, 2, 256, 512
    p = _routed_case(rng, t, e, k, h)
    wp = pack_int4(rng.integers(-8, 8, size=(e, 2 * inter, h)))
    ws = rng.uniform(0.002, 0.02, size=(e, 2 * inter, h // 128)).astype(np.float32)
    wd, sd = _prepack(fge, wp, ws, fmt, interleave=True)
    hq, hs = fge.grouped_gemm_w4a8(to_dev(p["aq"]), to_dev(p["as_"]), to_dev(p["offsets"]), wd,
                                   sd, fmt=_fmt(fge, fmt), epilogue="swiglu")
    c = oracle.grouped_gemm_w4a8(p["aq"], p["as_"], p["offsets"], wp, ws)
    rq, rs, _ = oracle.swiglu_requant(c, inter)
    gq, gs = host(hq), host(hs)
    np.testing.assert_allclose(gs, rs, rtol=1e-4)
    diff = gq != rq
    assert diff.mean() <= 0.005, diff.mean()
    assert np.all(np.abs(gq[diff].astype(int) - rq[diff].astype(int)) == 1)


# ------------------------------------------------------------------------ dense W8A8
def _dense_ref(fge, d):
    wq, sw = oracle.quant_act_per_tensor(d.w)
    return wq, sw


def test_w8a8_weight_quant_matches_oracle(fge):
    d = dense_inputs(16)
    wq_g, sw_g = fge.fp8_quant_act(bf16_dev(d.w_bits), "tensor")
    wq, sw = _dense_ref(fge, d)
    assert host(sw_g)[0] == sw and np.array_equal(host(wq_g), wq)


@pytest.mark.parametrize("m", [1, 16, 300, 2048])
def test_linear_w8a8(fge, m):
    d = dense_inputs(m)
    wq, sw = _dense_ref(fge, d)
    y = fge.linear_w8a8(bf16_dev(d.x_bits), to_dev(wq), to_dev(np.array([sw], np.float32)))
    xq, sa = oracle.quant_act_per_tensor(d.x)
    ref = oracle.linear_w8a8_gemm(xq, sa, wq, sw)
    absref = (float(sa) * float(sw)) * (np.abs(oracle.e4m3_decode(xq)) @ np.abs(oracle.e4m3_decode(wq)).T)
    check_gemm(host(y), ref, absref, True)


@pytest.mark.parametrize("m", [200, 1, 5, 16])
def test_gemm_w8a8_exact(fge, m):
    # m <= 16 runs the decode tile (weights on the 128-row side of the MMA, 16 token columns)
    rng = np.random.default_rng(51 + m)
    n, kdim = 384, 512
    a = rng.integers(-8, 9, size=(m, kdim)).astype(np.float32)
    w = rng.integers(-8, 9, size=(n, kdim)).astype(np.float32)
    aq, wq = oracle.e4m3_encode(a), oracle.e4m3_encode(w)
    sa, sw = np.float32(0.5), np.float32(2.0 ** -7)
    y = fge.gemm_w8a8(to_dev(aq), to_dev(np.array([sa])), to_dev(wq), to_dev(np.array([sw])),
                      out_dtype=torch.float32)
    ref = oracle.linear_w8a8_gemm(aq, sa, wq, sw)
    assert np.array_equal(host(y).astype(np.float64), ref)


@pytest.mark.parametrize("m", [1, 7, 16, 17])
def test_gemm_w8a8_rows_exact_decode_sizes(fge, m):
    # per-row activation scales (powers of two) on the decode tile: exact in float32
    rng = np.random.default_rng(77 + m)
    n, kdim = 256, 384
    a = rng.integers(-8, 9, size=(m, kdim)).astype(np.float32)
    w = rng.integers(-8, 9, size=(n, kdim)).astype(np.float32)
    aq, wq = oracle.e4m3_encode(a), oracle.e4m3_encode(w)
    sa = (2.0 ** rng.integers(-6, 3, size=m)).astype(np.float32)
    sw = np.float32(2.0 ** -5)
    y = fge.gemm_w8a8_rows(to_dev(aq), to_dev(sa), to_dev(wq), to_dev(np.array([sw])),
                           out_dtype=torch.float32)
    ref = oracle.linear_w8a8_rows_gemm(aq, sa, wq, sw)
    assert np.array_equal(host(y).astype(np.float64), ref)


# ------------------------------------------------------------------------ gathered A rows
@pytest.mark.parametrize("epi", ["store", "swiglu"])
@pytest.mark.parametrize("t,e,k,h,n", [(64, 8, 2, 256, 512), (300, 16, 4, 1024, 768),
                                       (1000, 64, 8, 2048, 1536)])
def test_gather_equals_permuted_copy(fge, epi, t, e, k, h, n):
    """The GEMM that gathers its A rows by row_token from the token-ordered activations gives
    exactly what the GEMM on the permuted copy gives (same operands, same arithmetic), with
    skewed routing (some experts empty, ragged tails)."""
    rng = np.random.default_rng(t + h)
    lg = (rng.standard_normal((t, e)) - 1.1 * np.log(np.arange(1, e + 1))).astype(np.float32)
    x = rng.standard_normal((t, h)).astype(np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    xq, xs = fge.fp8_quant_act(bf16_dev(bits), "g128")
    ids, _ = fge.moe_topk_gate(to_dev(lg), k)
    full = fge.moe_permute(ids, e, xq, xs)
    idx = fge.moe_permute(ids, e, xq, xs, index_only=True)
    for key in ("offsets", "row_token", "token_row"):
        assert torch.equal(full[key], idx[key])
    assert set(idx) == {"offsets", "row_token", "token_row"}
    wp = pack_int4(rng.integers(-8, 8, size=(e, n, h)))
    ws = rng.uniform(0.002, 0.02, size=(e, n, h // 128)).astype(np.float32)
    wd, sd = _prepack(fge, wp, ws, "subnormal", interleave=(epi == "swiglu"))
    a = fge.grouped_gemm_w4a8(full["aq"], full["as_"], full["offsets"], wd, sd, epilogue=epi)
    b = fge.grouped_gemm_w4a8_gather(xq, xs, idx["row_token"], idx["offsets"], wd, sd,
                                     epilogue=epi)
    if epi == "swiglu":
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    else:
        assert torch.equal(a, b)
    # and against the oracle on the same quantized operands
    if epi == "store" and t <= 300:
        p = {kk: host(full[kk]) for kk in ("aq", "as_", "offsets")}
        ref = oracle.grouped_gemm_w4a8(p["aq"], p["as_"], p["offsets"], wp, ws)
        absref = abs_grouped(p["aq"], p["as_"], p["offsets"], wp, ws)
        check_gemm(host(b), ref, absref, False)


@pytest.mark.parametrize("t,e,k,n", [(1024, 4, 1, 768), (700, 3, 2, 768), (700, 3, 2, 640)])
def test_grouped_bf16_full_and_ragged_tiles(fge, t, e, k, n):
    """bf16 output with many full 128-row tiles (each warp stages its rows in shared memory
    and writes them with TMA tile stores) next to each expert's ragged last tile (stored
    directly).  N = 640 takes the 128-column tile (N not a multiple of 256)."""
    rng = np.random.default_rng(t + e + n)
    h = 512
    p = _routed_case(rng, t, e, k, h)
    assert np.diff(p["offsets"]).max() >= 256
    q = rng.integers(-8, 8, size=(e, n, h))
    wp = pack_int4(q)
    ws = rng.uniform(0.002, 0.02, size=(e, n, h // 128)).astype(np.float32)
    wd, sd = _prepack(fge, wp, ws, "subnormal")
    out = fge.grouped_gemm_w4a8(to_dev(p["aq"]), to_dev(p["as_"]), to_dev(p["offsets"]), wd, sd,
                                out_dtype=torch.bfloat16)
    ref = oracle.grouped_gemm_w4a8(p["aq"], p["as_"], p["offsets"], wp, ws)
    absref = abs_grouped(p["aq"], p["as_"], p["offsets"], wp, ws)
    check_gemm(host(out), ref, absref, True)


def test_swiglu_full_and_ragged_tiles(fge):
    """SwiGLU + requant epilogue with full 128-row tiles (TMA tile stores of the codes) and
    ragged last tiles (direct stores)."""
    rng = np.random.default_rng(77)
    t, e, k, h, inter = 1024, 4, 1, 256, 512
    p = _routed_case(rng, t, e, k, h)
    assert np.diff(p["offsets"]).max() >= 256
    wp = pack_int4(rng.integers(-8, 8, size=(e, 2 * inter, h)))
    ws = rng.uniform(0.002, 0.02, size=(e, 2 * inter, h // 128)).astype(np.float32)
    wd, sd = _prepack(fge, wp, ws, "subnormal", interleave=True)
    hq, hs = fge.grouped_gemm_w4a8(to_dev(p["aq"]), to_dev(p["as_"]), to_dev(p["offsets"]), wd,
                                   sd, epilogue="swiglu")
    c = oracle.grouped_gemm_w4a8(p["aq"], p["as_"], p["offsets"], wp, ws)
    rq, rs, _ = oracle.swiglu_requant(c, inter)
    gq, gs = host(hq), host(hs)
    np.testing.assert_allclose(gs, rs, rtol=1e-4)
    diff = gq != rq
    assert diff.mean() <= 0.005, diff.mean()
    assert np.all(np.abs(gq[diff].astype(int) - rq[diff].astype(int)) == 1)
