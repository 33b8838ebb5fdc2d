"""Pins for the single-threaded C++ oracle (``oracle/oracle_ref.cpp``).

The C++ restatement and the numpy one were written separately and share no code; where a
rule can be written two ways they take different routes (bit manipulation against
frexp/rint for the e4m3 and bf16 roundings, repeated maximum against a sort for top-k), so
agreement between them is a check on both.  Beside that cross-check the C++ oracle is pinned
on its own: the encoder against a brute-force nearest-value search over every float32 of
the e4m3 range, the hand-derived e4m3 code points, exact GEMM cases and closed forms.
"""

from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import native as cpp
from workloads import moe_inputs, pack_int4


def test_decode_table_equals_numpy_and_hand_values():
    tab = cpp.e4m3_decode_table()
    ref = oracle.e4m3_decode_table()
    assert np.array_equal(np.isnan(tab), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(tab[ok], ref[ok])
    # hand-derived: 0x08 = 2^-6, 0x01 = 2^-9, 0x7E = 1.75 * 2^8 = 448, 0x38 = 1, 0xC0 = -2
    assert (tab[0x08], tab[0x01], tab[0x7E], tab[0x38], tab[0xC0]) == (2 ** -6, 2 ** -9, 448.0,
                                                                       1.0, -2.0)
    assert np.isnan(tab[0x7F]) and np.isnan(tab[0xFF])


def test_encode_brute_force_every_float_of_the_range():
    # every float32 in [2^-12, 2^10), both signs: below 2^-10 everything rounds to zero and
    # above 464 everything saturates, so this covers every rounding decision of the format
    assert cpp.encode_selfcheck(-12, 10) == 0


def test_encode_equals_numpy_on_bf16_values_and_random_floats():
    bits = np.arange(65536, dtype=np.uint32) << 16
    v = bits.view(np.float32)
    v = v[np.isfinite(v)]
    for scale in (1.0, 2.0 ** -7, 2.0 ** 5, 0.37):
        with np.errstate(over="ignore"):
            x = (v * np.float32(scale)).astype(np.float32)
        x = x[np.isfinite(x)]
        assert np.array_equal(cpp.e4m3_encode(x), oracle.e4m3_encode(x))
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(1 << 20) * np.exp(rng.uniform(-14, 8, 1 << 20))).astype(np.float32)
    assert np.array_equal(cpp.e4m3_encode(x), oracle.e4m3_encode(x))
    tiny = np.array([0.0, -0.0, 1e-45, -1e-45, 2.0 ** -10, 2.0 ** -10 * 1.0000001, 1e30, -1e30,
                     np.inf, -np.inf], np.float32)
    assert np.array_equal(cpp.e4m3_encode(tiny), oracle.e4m3_encode(tiny))
    assert cpp.e4m3_encode(np.float32(-0.0)).item() == 0x80


def test_encode_matches_torch_cast_in_range():
    rng = np.random.default_rng(1)
    x = (rng.uniform(-448, 448, 200000)).astype(np.float32)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(cpp.e4m3_encode(x), want)


def test_bf16_round_equals_numpy_and_torch():
    rng = np.random.default_rng(2)
    v = rng.standard_normal(200000) * np.exp(rng.uniform(-85, 85, 200000))
    v = np.concatenate([v, [0.0, -0.0, 2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -134, 1 + 2.0 ** -8,
                            1 + 3 * 2.0 ** -8, 1 + 2.0 ** -8 + 2.0 ** -40]])
    assert np.array_equal(cpp.bf16_round(v), oracle.bf16_round(v))
    f = rng.standard_normal(100000).astype(np.float32)
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(cpp.bf16_round(f.astype(np.float64)), want)
    # one rounding from float64: 1 + 2^-8 + 2^-40 lies just above the tie, so it rounds up,
    # where rounding through float32 first would land on the tie and go to even (down)
    assert cpp.bf16_round(np.array([1 + 2.0 ** -8 + 2.0 ** -40])).item() == 0x3F81


@pytest.mark.parametrize("mode", ["g128", "tensor", "row"])
def test_quantizers_equal_numpy(mode):
    inp = moe_inputs("tiny", seed=3)
    x = np.concatenate([inp.x, np.zeros((2, inp.H), np.float32),
                        np.full((1, inp.H), 1e-40, np.float32)])
    fn_c = dict(g128=cpp.quant_act_g128, tensor=cpp.quant_act_per_tensor,
                row=cpp.quant_act_per_row)[mode]
    fn_n = dict(g128=oracle.quant_act_g128, tensor=oracle.quant_act_per_tensor,
                row=oracle.quant_act_per_row)[mode]
    qc, sc = fn_c(x)
    qn, sn = fn_n(x)
    assert np.array_equal(qc, qn)
    assert np.array_equal(np.asarray(sc), np.asarray(sn))


def test_quant_closed_form_group():
    # x = c * (1..128): amax = 128c, s = fp32(128c/448); the value 128c encodes to 448
    c = np.float32(0.5)
    x = (c * np.arange(1, 129, dtype=np.float32))[None, :]
    q, s = cpp.quant_act_g128(x)
    assert s[0, 0] == np.float32(np.float32(64.0) / np.float32(448.0))
    assert q[0, 127] == 0x7E
    q0, s0 = cpp.quant_act_g128(np.zeros((1, 128), np.float32))
    assert s0[0, 0] == 1.0 and not q0.any()


def test_topk_equals_numpy_and_ties():
    rng = np.random.default_rng(4)
    lg = rng.standard_normal((300, 64)).astype(np.float32)
    lg[::7, 3] = lg[::7, 9]                       # exact ties between two experts
    for k in (1, 2, 8, 64):
        ic, gc = cpp.topk_gate(lg, k)
        i_n, g_n = oracle.topk_gate(lg, k)
        assert np.array_equal(ic, i_n)
        assert np.allclose(gc, g_n, rtol=2e-7, atol=0)
    ids, gates = cpp.topk_gate(np.zeros((2, 16), np.float32), 4)
    assert ids.tolist() == [[0, 1, 2, 3]] * 2 and np.all(gates == np.float32(0.25))


def test_permute_equals_numpy_and_invariants():
    rng = np.random.default_rng(5)
    t, e, k, h = 257, 12, 3, 256
    ids = np.stack([rng.choice(e - 2, size=k, replace=False) for _ in range(t)]).astype(np.int32)
    xq = rng.integers(0, 256, size=(t, h), dtype=np.uint8)
    xs = rng.uniform(0.1, 1, size=(t, h // 128)).astype(np.float32)
    pc = cpp.moe_permute(ids, e, xq, xs)
    pn = oracle.moe_permute(ids, e, xq, xs)
    for key in ("counts", "offsets", "row_token", "token_row", "aq", "as_"):
        assert np.array_equal(pc[key], pn[key]), key
    assert pc["counts"].sum() == t * k and pc["counts"][-2:].sum() == 0
    assert np.array_equal(pc["row_token"][pc["token_row"]], np.repeat(np.arange(t), k).reshape(t, k))


def _exact_gemm_case(seed):
    # small-integer e4m3 activations and power-of-two scales: every partial sum is exact
    rng = np.random.default_rng(seed)
    e, n, kdim, rows = 3, 48, 256, 40
    counts = np.array([17, 0, 23])
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    avals = rng.integers(-16, 17, size=(rows, kdim))
    aq = oracle.e4m3_encode(avals.astype(np.float32))
    as_ = np.ldexp(1.0, rng.integers(-4, 3, size=(rows, kdim // 128))).astype(np.float32)
    q = rng.integers(-8, 8, size=(e, n, kdim))
    sw = np.ldexp(1.0, rng.integers(-6, 0, size=(e, n, kdim // 128))).astype(np.float32)
    return avals, aq, as_, offsets, q, sw


def test_grouped_gemm_exact_case_against_fractions():
    avals, aq, as_, offsets, q, sw = _exact_gemm_case(6)
    got = cpp.grouped_gemm_w4a8(aq, as_, offsets, pack_int4(q), sw)
    for r in (0, 5, 16, 17, 30, 39):
        e = int(np.searchsorted(offsets, r, side="right") - 1)
        for n in (0, 7, 47):
            want = Fraction(0)
            for g in range(2):
                part = sum(int(avals[r, kk]) * int(q[e, n, kk]) for kk in range(g * 128, g * 128 + 128))
                want += Fraction(float(as_[r, g])) * Fraction(float(sw[e, n, g])) * part
            assert Fraction(got[r, n]) == want


def test_grouped_gemm_equals_numpy_bit_for_bit():
    inp = moe_inputs("tiny", seed=7)
    xq, xs = oracle.quant_act_g128(inp.x)
    ids, _ = oracle.topk_gate(inp.logits, inp.k)
    p = oracle.moe_permute(ids, inp.E, xq, xs)
    got = cpp.grouped_gemm_w4a8(p["aq"], p["as_"], p["offsets"], inp.w_gu, inp.s_gu)
    want = oracle.grouped_gemm_w4a8(p["aq"], p["as_"], p["offsets"], inp.w_gu, inp.s_gu)
    assert np.array_equal(got, want)


def test_grouped_gemm_all_ones_closed_form():
    e, n, kdim, rows = 2, 16, 384, 9
    offsets = np.array([0, 4, 9], np.int32)
    aq = np.full((rows, kdim), 0x38, np.uint8)                    # e4m3 1.0
    as_ = np.random.default_rng(8).uniform(0.5, 2, (rows, 3)).astype(np.float32)
    sw = np.random.default_rng(9).uniform(0.002, 0.02, (e, n, 3)).astype(np.float32)
    w = pack_int4(np.ones((e, n, kdim), np.int8))
    got = cpp.grouped_gemm_w4a8(aq, as_, offsets, w, sw)
    for r in range(rows):
        ex = 0 if r < 4 else 1
        want = sum(128.0 * float(as_[r, g]) * float(sw[ex, :, g][0]) for g in range(3))
        assert abs(got[r, 0] - want) <= 1e-12 * abs(want)


def test_swiglu_and_combine_equal_numpy():
    rng = np.random.default_rng(10)
    c = rng.standard_normal((70, 512)) * 3
    hq_c, hs_c, h_c = cpp.swiglu_requant(c, 256)
    hq_n, hs_n, h_n = oracle.swiglu_requant(c, 256)
    # CPU exp implementations may differ in the last bit of a float64; after the float32
    # rounding of h that shows at most as one float32 step, and almost never
    diff = h_c != h_n
    assert diff.mean() < 1e-3
    assert np.all(np.abs(h_c - h_n) <= np.spacing(np.abs(h_n)))
    assert (hq_c != hq_n).mean() < 1e-3 and (hs_c != hs_n).mean() < 1e-2
    y = rng.standard_normal((60, 128)).astype(np.float32)
    token_row = rng.permutation(60).reshape(20, 3).astype(np.int32)
    gates = rng.uniform(0, 1, (20, 3)).astype(np.float32)
    assert np.array_equal(cpp.moe_combine(y, token_row, gates),
                          oracle.moe_combine(y, token_row, gates))


def test_w8a8_equals_numpy_and_exact_case():
    rng = np.random.default_rng(11)
    a = oracle.e4m3_encode(rng.integers(-16, 17, (9, 256)).astype(np.float32))
    w = oracle.e4m3_encode(rng.integers(-16, 17, (24, 256)).astype(np.float32))
    got = cpp.linear_w8a8_gemm(a, np.float32(0.25), w, np.float32(0.125))
    ints = oracle.e4m3_decode(a) @ oracle.e4m3_decode(w).T
    assert np.array_equal(got, ints / 32.0)
    wq, sw = oracle.quant_act_per_tensor(rng.standard_normal((24, 256)).astype(np.float32) * 0.02)
    aq, sa = oracle.quant_act_per_tensor(rng.standard_normal((9, 256)).astype(np.float32))
    assert np.array_equal(cpp.linear_w8a8_gemm(aq, sa, wq, sw),
                          oracle.linear_w8a8_gemm(aq, sa, wq, sw))
    rows = rng.uniform(0.01, 1, 9).astype(np.float32)
    assert np.array_equal(cpp.linear_w8a8_gemm(aq, 0.0, wq, sw, sa_rows=rows),
                          oracle.linear_w8a8_rows_gemm(aq, rows, wq, sw))


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_tiny_layer_equals_numpy(out_dtype):
    inp = moe_inputs("tiny", seed=12)
    got = cpp.moe_layer_forward(inp.logits, inp.x, inp.k, inp.w_gu, inp.s_gu, inp.w_dn,
                                inp.s_dn, inp.I, out_dtype=out_dtype)
    want, _ = oracle.moe_layer_forward(inp.logits, inp.x, inp.k, inp.w_gu, inp.s_gu, inp.w_dn,
                                       inp.s_dn, inp.I, out_dtype=out_dtype)
    # identical except where a last-bit exp difference flips a SwiGLU requant code
    rel = np.linalg.norm(got - want) / np.linalg.norm(want)
    assert rel < 1e-5, rel
    assert np.mean(got != want) < 0.02


def test_mx_quant_equals_numpy_over_every_bf16_value():
    bits = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    v = bits[np.isfinite(bits)]
    v = np.concatenate([v, np.zeros((-v.size) % 1024, np.float32)]).reshape(-1, 1024)
    rng = np.random.default_rng(13)
    v = v[:, rng.permutation(1024)]             # mix magnitudes inside each 32-value block
    pc, sc = cpp.mx_quant_e2m1(v)
    pn, sn = oracle.mx_quant_e2m1(v.astype(np.float64))
    assert np.array_equal(pc, pn) and np.array_equal(sc, sn)
    zero = np.zeros((1, 64), np.float32)
    assert np.array_equal(cpp.mx_quant_e2m1(zero)[1], np.zeros((1, 2), np.uint8))


def test_stack_helpers_equal_numpy():
    rng = np.random.default_rng(14)
    h = (rng.standard_normal((9, 256)) * 3).astype(np.float32)
    assert np.array_equal(cpp.rmsnorm(h), oracle.rmsnorm(h))
    xn = oracle.rmsnorm(h)
    w = (rng.standard_normal((16, 256)) * 0.02).astype(np.float32)
    got, want = cpp.router_logits(xn, w), oracle.router_logits(xn, w)
    # float64 sums in two orders, then one float32 rounding: at most one float32 step apart
    assert np.all(np.abs(got - want) <= np.spacing(np.abs(want)))
    v = rng.standard_normal((5, 4 * 128)).astype(np.float32)
    assert np.array_equal(cpp.identity_attention(v, 16, 4), oracle.identity_attention(v, 16, 4))


@pytest.mark.parametrize("rows", [False, True])
def test_dense_projection_equals_numpy(rows):
    rng = np.random.default_rng(15)
    wq, sw = oracle.quant_act_per_tensor((rng.standard_normal((40, 256)) * 0.02).astype(np.float32))
    x = rng.standard_normal((7, 256)).astype(np.float32)
    x[3] *= 20
    want = (oracle.linear_w8a8_rows if rows else oracle.linear_w8a8)(x, wq, sw)[0]
    assert np.array_equal(cpp.linear_w8a8(x, wq, sw, rows=rows), want)


def test_int4_baseline_equals_numpy():
    inp = moe_inputs("tiny", seed=16)
    rows = np.arange(12)
    got = cpp.moe_layer_int4_baseline(inp.logits[rows], inp.x[rows], inp.k, inp.w_gu, inp.s_gu,
                                      inp.w_dn, inp.s_dn, inp.I, out_dtype="f32")
    want, _ = oracle.moe_layer_int4_baseline(inp.logits[rows], inp.x[rows], inp.k, inp.w_gu,
                                             inp.s_gu, inp.w_dn, inp.s_dn, inp.I, out_dtype="f32")
    assert np.allclose(got, want, rtol=1e-6, atol=1e-6 * np.abs(want).max())


def test_stacked_prefill_equals_numpy():
    rng = np.random.default_rng(17)
    T, H, E, I, k, nh, nkv = 24, 256, 8, 256, 2, 2, 1
    layers = []
    for _ in range(3):
        wv, sv = oracle.quant_act_per_tensor((rng.standard_normal((nkv * 128, H)) * 0.02).astype(np.float32))
        wo, so = oracle.quant_act_per_tensor((rng.standard_normal((H, nh * 128)) * 0.02).astype(np.float32))
        layers.append(dict(
            wv=wv, sv=sv, wo=wo, so=so,
            w_router=(rng.standard_normal((E, H)) * 0.02).astype(np.float32),
            w_gu=pack_int4(rng.integers(-8, 8, (E, 2 * I, H))),
            s_gu=rng.uniform(0.0005, 0.002, (E, 2 * I, H // 128)).astype(np.float32),
            w_dn=pack_int4(rng.integers(-8, 8, (E, H, I))),
            s_dn=rng.uniform(0.0005, 0.002, (E, H, I // 128)).astype(np.float32)))
    h0 = rng.standard_normal((T, H)).astype(np.float32)
    hc, rc = cpp.stacked_prefill(h0, layers, k, I, nh, nkv)
    hn, rn = oracle.stacked_prefill(h0, layers, k, I, nh, nkv)
    # the router sums and the SwiGLU exp may differ in a last bit between the two, which
    # can move a requant code; everything else is the same arithmetic
    cos = float((hc.ravel().astype(np.float64) @ hn.ravel()) /
                np.sqrt((hc.astype(np.float64) ** 2).sum() * (hn.astype(np.float64) ** 2).sum()))
    assert cos >= 0.99999, cos
    assert all(np.array_equal(a, b) for a, b in zip(rc, rn))


def test_mx_grouped_gemm_equals_numpy():
    # the C++ restatement (E2M1 values from their fields, ldexp scaling, per-element loops)
    # against the numpy one (decode table, dequantized matrix, matmul per group), routed rows
    # with an empty expert and block scales spread over several binades
    rng = np.random.default_rng(17)
    counts = [40, 0, 23, 1]
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    r, k, n = int(offsets[-1]), 384, 48
    codes = rng.integers(0, 256, (r, k // 2)).astype(np.uint8)
    scales = rng.integers(115, 140, (r, k // 32)).astype(np.uint8)
    q = rng.integers(-8, 8, (4, n, k))
    wp = (q[..., 0::2] & 0xF | (q[..., 1::2] & 0xF) << 4).astype(np.uint8)
    sw = rng.uniform(0.002, 0.02, (4, n, k // 128)).astype(np.float32)
    got = cpp.grouped_gemm_mxf4_w4(codes, scales, offsets, wp, sw)
    ref = oracle.grouped_gemm_mxf4_w4(codes, scales, offsets, wp, sw)
    assert np.array_equal(got, ref)
