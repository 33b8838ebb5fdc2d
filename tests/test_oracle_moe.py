"""Pins for the oracle's routing, permutation, grouped W4A8 GEMM, SwiGLU requant, combine,
dense W8A8 GEMM and stacked-layer helpers.

Expected values come from closed forms, exact integer arithmetic (Python ints and
fractions), a deliberately naive element-by-element loop, library routines (scipy softmax,
torch silu) or invariants -- never from the oracle itself.
"""

from fractions import Fraction

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from workloads import moe_inputs, pack_int4


# --- top-k gate --------------------------------------------------------------------------

def test_topk_with_k_equal_E_is_plain_softmax():
    rng = np.random.default_rng(10)
    lg = rng.standard_normal((50, 8)).astype(np.float32)
    ids, gates = oracle.topk_gate(lg, 8)
    order = np.argsort(-lg.astype(np.float64), axis=1, kind="stable")
    assert np.array_equal(ids, order)
    sm = scipy.special.softmax(lg.astype(np.float64), axis=1)
    assert np.allclose(gates, np.take_along_axis(sm, order, 1), rtol=1e-6, atol=0)


def test_topk_ties_choose_lower_ids_and_equal_gates():
    lg = np.zeros((3, 16), np.float32)
    ids, gates = oracle.topk_gate(lg, 4)
    assert ids.tolist() == [[0, 1, 2, 3]] * 3
    assert np.all(gates == np.float32(0.25))
    lg2 = np.array([[1, 5, 5, 0, 5]], np.float32)
    ids2, _ = oracle.topk_gate(lg2, 2)
    assert ids2.tolist() == [[1, 2]]


def test_topk_gates_renormalise_full_softmax():
    rng = np.random.default_rng(11)
    lg = rng.standard_normal((40, 64)).astype(np.float32)
    ids, gates = oracle.topk_gate(lg, 8)
    sm = scipy.special.softmax(lg.astype(np.float64), axis=1)
    sel = np.take_along_axis(sm, ids.astype(np.int64), 1)
    assert np.allclose(gates, sel / sel.sum(1, keepdims=True), rtol=1e-6, atol=0)
    assert np.all(np.diff(np.take_along_axis(lg, ids.astype(np.int64), 1), axis=1) <= 0)


# --- permute -----------------------------------------------------------------------------

def _perm_case(t=300, e=12, k=3, h=256, seed=12):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.choice(e, size=k, replace=False) for _ in range(t)]).astype(np.int32)
    xq = rng.integers(0, 256, size=(t, h), dtype=np.uint8)
    xs = rng.uniform(0.1, 1, size=(t, h // 128)).astype(np.float32)
    return ids, xq, xs


def test_permute_invariants():
    ids, xq, xs = _perm_case()
    t, k = ids.shape
    p = oracle.moe_permute(ids, 12, xq, xs)
    assert p["counts"].sum() == t * k
    assert np.array_equal(p["counts"], np.bincount(ids.ravel(), minlength=12))
    assert p["offsets"][0] == 0 and np.array_equal(np.diff(p["offsets"]), p["counts"])
    assert np.array_equal(np.bincount(p["row_token"], minlength=t), np.full(t, k))
    rows = p["token_row"].ravel()
    assert np.array_equal(np.sort(rows), np.arange(t * k))
    assert np.array_equal(p["row_token"][p["token_row"]], np.repeat(np.arange(t)[:, None], k, 1))
    for e in range(12):
        seg = p["row_token"][p["offsets"][e]:p["offsets"][e + 1]]
        assert np.all(np.diff(seg) > 0)                       # stable: token order kept
        assert all(e in ids[tok] for tok in seg)
    for tok in range(t):
        for j in range(k):
            r = p["token_row"][tok, j]
            assert p["offsets"][ids[tok, j]] <= r < p["offsets"][ids[tok, j] + 1]
    assert np.array_equal(p["aq"], xq[p["row_token"]])
    assert np.array_equal(p["as_"], xs[p["row_token"]])


def test_permute_empty_experts_and_single_expert():
    ids = np.zeros((5, 1), np.int32) + 3
    xq = np.arange(5 * 128, dtype=np.uint8).reshape(5, 128)
    xs = np.ones((5, 1), np.float32)
    p = oracle.moe_permute(ids, 6, xq, xs)
    assert p["offsets"].tolist() == [0, 0, 0, 0, 5, 5, 5]
    assert p["row_token"].tolist() == [0, 1, 2, 3, 4]


# --- grouped W4A8 GEMM -------------------------------------------------------------------

def _naive_grouped(aq, as_, offsets, w_packed, w_scale):
    """Element-by-element loop with every value decoded on its own (independent of the
    vectorised oracle): decode e4m3 by its bit fields, int4 by its nibbles."""
    def dec(c):
        s = -1.0 if c & 0x80 else 1.0
        e, m = (c >> 3) & 15, c & 7
        return s * (m / 8 * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))

    def nib(b, hi):
        v = (b >> 4) if hi else (b & 15)
        return v - 16 if v >= 8 else v

    r_tot, kdim = aq.shape
    n = w_packed.shape[1]
    out = np.zeros((r_tot, n))
    for e in range(len(offsets) - 1):
        for r in range(offsets[e], offsets[e + 1]):
            for col in range(n):
                tot = 0.0
                for g in range(kdim // 128):
                    part = 0.0
                    for kk in range(g * 128, (g + 1) * 128):
                        part += dec(int(aq[r, kk])) * nib(int(w_packed[e, col, kk // 2]), kk % 2)
                    tot += float(as_[r, g]) * float(w_scale[e, col, g]) * part
                out[r, col] = tot
    return out


def test_grouped_gemm_matches_naive_loop_on_tiny_case():
    rng = np.random.default_rng(13)
    e, n, kdim = 3, 5, 256
    offsets = np.array([0, 2, 2, 5], np.int32)               # expert 1 is empty
    aq = rng.integers(0, 256, size=(6, kdim), dtype=np.uint8)
    aq[(aq & 0x7F) == 0x7F] = 0x11                            # no NaN codes
    as_ = rng.uniform(0.01, 1, size=(6, 2)).astype(np.float32)
    wp = rng.integers(0, 256, size=(e, n, kdim // 2), dtype=np.uint8)
    ws = rng.uniform(0.002, 0.02, size=(e, n, 2)).astype(np.float32)
    got = oracle.grouped_gemm_w4a8(aq, as_, offsets, wp, ws)
    ref = _naive_grouped(aq, as_, offsets, wp, ws)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-300)
    assert np.all(got[5] == 0)                                 # row past offsets[E]


def test_grouped_gemm_exact_small_integer_case():
    # integer activations |a| <= 16 and power-of-two scales: the result is an exact dyadic
    # rational, computed here with Python integers and Fractions.
    rng = np.random.default_rng(14)
    e, n, kdim, r = 2, 7, 384, 9
    a_int = rng.integers(-16, 17, size=(r, kdim))
    aq = oracle.e4m3_encode(a_int.astype(np.float32))
    q = rng.integers(-8, 8, size=(e, n, kdim))
    wp = pack_int4(q)
    as_ = np.ldexp(1.0, rng.integers(-8, 4, size=(r, 3))).astype(np.float32)
    ws = np.ldexp(1.0, rng.integers(-10, -4, size=(e, n, 3))).astype(np.float32)
    offsets = np.array([0, 4, 9], np.int32)
    got = oracle.grouped_gemm_w4a8(aq, as_, offsets, wp, ws)
    for row in range(r):
        ex = 0 if row < 4 else 1
        for col in range(n):
            tot = Fraction(0)
            for g in range(3):
                s = sum(int(a_int[row, kk]) * int(q[ex, col, kk]) for kk in range(g * 128, g * 128 + 128))
                tot += Fraction(float(as_[row, g])) * Fraction(float(ws[ex, col, g])) * s
            assert got[row, col] == float(tot)


def test_grouped_gemm_all_ones_closed_form():
    # a = 1.0 (code 0x38), every weight nibble = 1 -> C[r, n] = sum_g 128 * as[r,g] * sw[e,n,g]
    rng = np.random.default_rng(15)
    r, n, kdim = 6, 4, 512
    aq = np.full((r, kdim), 0x38, np.uint8)
    wp = np.full((2, n, kdim // 2), 0x11, np.uint8)
    as_ = rng.uniform(0.1, 2, size=(r, 4)).astype(np.float32)
    ws = rng.uniform(0.002, 0.02, size=(2, n, 4)).astype(np.float32)
    offsets = np.array([0, 3, 6], np.int32)
    got = oracle.grouped_gemm_w4a8(aq, as_, offsets, wp, ws)
    for row in range(r):
        ex = 0 if row < 3 else 1
        ref = 128 * (as_[row].astype(np.float64)[None, :] * ws[ex].astype(np.float64)).sum(1)
        assert np.allclose(got[row], ref, rtol=1e-14)


def test_grouped_gemm_one_scale_equals_per_tensor_formula():
    # all group scales equal -> the grouped GEMM is the per-tensor W8A8 formula with the
    # int4 weights written as e4m3 codes (int4 is exact in e4m3)
    rng = np.random.default_rng(16)
    r, n, kdim = 10, 6, 256
    aq = oracle.e4m3_encode(rng.standard_normal((r, kdim)).astype(np.float32) * 30)
    q = rng.integers(-8, 8, size=(1, n, kdim))
    sa, sw = np.float32(0.037), np.float32(0.0061)
    got = oracle.grouped_gemm_w4a8(aq, np.full((r, 2), sa), np.array([0, r]), pack_int4(q),
                                   np.full((1, n, 2), sw))
    ref = oracle.linear_w8a8_gemm(aq, sa, oracle.e4m3_encode(q[0].astype(np.float32)), sw)
    assert np.allclose(got, ref, rtol=1e-13)


# --- W8A8 --------------------------------------------------------------------------------

def test_w8a8_exact_power_of_two_case():
    rng = np.random.default_rng(17)
    a = rng.integers(-12, 13, size=(5, 256))
    w = rng.integers(-12, 13, size=(7, 256))
    got = oracle.linear_w8a8_gemm(oracle.e4m3_encode(a.astype(np.float32)), np.float32(0.25),
                                  oracle.e4m3_encode(w.astype(np.float32)), np.float32(2.0 ** -7))
    assert np.array_equal(got, (a @ w.T) * 2.0 ** -9)


# --- SwiGLU requant and combine ------------------------------------------------------------

def test_swiglu_closed_forms_and_library_silu():
    rng = np.random.default_rng(18)
    c = rng.standard_normal((4, 512)) * 3
    c[0, :256] = 0.0                                            # silu(0) = 0
    hq, hs, h = oracle.swiglu_requant(c, 256)
    # 0 * u keeps the sign of u, so the codes are +-0 (0x00 / 0x80)
    assert np.all(h[0] == 0) and np.all(hq[0] & 0x7F == 0) and np.all(hs[0] == 1.0)
    c32 = torch.tensor(c.astype(np.float32).astype(np.float64))
    ref = (torch.nn.functional.silu(c32[:, :256]) * c32[:, 256:]).to(torch.float32).numpy()
    assert np.allclose(h, ref, rtol=2e-7, atol=0)
    q2, s2 = oracle.quant_act_g128(h)
    assert np.array_equal(q2, hq) and np.array_equal(s2, hs)


def test_combine_k1_gate1_is_inverse_permutation():
    rng = np.random.default_rng(19)
    ids = rng.integers(0, 5, size=(40, 1)).astype(np.int32)
    p = oracle.moe_permute(ids, 5, np.zeros((40, 128), np.uint8), np.ones((40, 1), np.float32))
    y = rng.standard_normal((40, 9))
    out = oracle.moe_combine(y, p["token_row"], np.ones((40, 1), np.float32))
    assert np.array_equal(out, y[p["token_row"][:, 0]])


def test_combine_linear_in_gates():
    rng = np.random.default_rng(20)
    tr = np.array([[0, 3], [1, 2]])
    y = rng.standard_normal((4, 5))
    g = np.array([[0.25, 0.75], [0.5, 0.5]], np.float32)
    out = oracle.moe_combine(y, tr, g)
    assert np.allclose(out[0], 0.25 * y[0] + 0.75 * y[3], rtol=1e-15)
    assert np.allclose(out[1], 0.5 * y[1] + 0.5 * y[2], rtol=1e-15)


# --- layer and stack helpers --------------------------------------------------------------

def test_tiny_layer_runs_and_is_deterministic():
    inp = moe_inputs("tiny", seed=3)
    args = (inp.logits, inp.x, inp.k, inp.w_gu, inp.s_gu, inp.w_dn, inp.s_dn, inp.I, inp.out)
    out1, d1 = oracle.moe_layer_forward(*args)
    out2, _ = oracle.moe_layer_forward(*args)
    assert out1.shape == (inp.T, inp.H) and np.array_equal(out1, out2)
    assert d1["offsets"][-1] == inp.T * inp.k and np.all(np.isfinite(out1))


def test_rmsnorm_closed_form_and_identity_attention():
    h = np.full((2, 256), 3.0, np.float32)
    h[1] = -0.5
    r = oracle.rmsnorm(h)
    assert np.all(r[0] == oracle.bf16_bits_to_f32(oracle.bf16_round(3 / np.sqrt(9 + 1e-6))))
    assert np.all(r[1] == oracle.bf16_bits_to_f32(oracle.bf16_round(-0.5 / np.sqrt(0.25 + 1e-6))))
    v = np.arange(2 * 512).reshape(2, 512).astype(np.float32)
    a = oracle.identity_attention(v, 16, 4)
    assert a.shape == (2, 2048)
    for head in range(16):
        assert np.array_equal(a[:, head * 128:(head + 1) * 128],
                              v[:, (head // 4) * 128:(head // 4 + 1) * 128])


# --- per-token int4 baseline ------------------------------------------------------------

def test_dequant_bank_matches_grouped_gemm_on_exact_activations():
    # integer activations (exact in e4m3) with unit activation scales: the grouped GEMM's
    # definition and a plain matmul with the dequantized bank must agree
    rng = np.random.default_rng(71)
    e, n, kdim, r = 2, 6, 256, 5
    a = rng.integers(-16, 17, size=(r, kdim)).astype(np.float32)
    q = rng.integers(-8, 8, size=(e, n, kdim))
    ws = rng.uniform(0.002, 0.02, size=(e, n, 2)).astype(np.float32)
    wp = pack_int4(q)
    offs = np.array([0, 3, 5], np.int32)
    got = oracle.grouped_gemm_w4a8(oracle.e4m3_encode(a), np.ones((r, 2), np.float32), offs,
                                   wp, ws)
    w = oracle.dequant_int4_bank(wp, ws, kdim)
    ref = np.concatenate([a[:3].astype(np.float64) @ w[0].T, a[3:].astype(np.float64) @ w[1].T])
    assert np.allclose(got, ref, rtol=1e-13)
    assert np.array_equal(w[1, 2, :128], q[1, 2, :128] * float(ws[1, 2, 0]))


def test_int4_baseline_single_expert_closed_form():
    # one expert, k = 1: the baseline is the expert FFN on each token with gate 1
    rng = np.random.default_rng(72)
    t, h, inter = 4, 128, 128
    x = rng.standard_normal((t, h)).astype(np.float32)
    q_gu = rng.integers(-8, 8, size=(1, 2 * inter, h))
    q_dn = rng.integers(-8, 8, size=(1, h, inter))
    s_gu = np.full((1, 2 * inter, 1), 0.01, np.float32)
    s_dn = np.full((1, h, 1), 0.02, np.float32)
    out, ids = oracle.moe_layer_int4_baseline(np.zeros((t, 1), np.float32), x, 1, pack_int4(q_gu),
                                              s_gu, pack_int4(q_dn), s_dn, inter, out_dtype="f32")
    c = x.astype(np.float64) @ (q_gu[0] * 0.01).T
    hh = c[:, :inter] / (1 + np.exp(-c[:, :inter])) * c[:, inter:]
    ref = hh @ (q_dn[0] * float(np.float32(0.02))).T
    assert np.all(ids == 0)
    assert np.allclose(out, ref.astype(np.float32), rtol=1e-6)


# --- W8A8 with row-wise activation scales ----------------------------------------------------

def test_w8a8_rows_equal_scales_is_per_tensor():
    rng = np.random.default_rng(31)
    aq = oracle.e4m3_encode(rng.standard_normal((9, 256)).astype(np.float32) * 40)
    wq = oracle.e4m3_encode(rng.standard_normal((5, 256)).astype(np.float32) * 40)
    sa, sw = np.float32(0.0173), np.float32(0.00091)
    got = oracle.linear_w8a8_rows_gemm(aq, np.full(9, sa, dtype=np.float32), wq, sw)
    ref = oracle.linear_w8a8_gemm(aq, sa, wq, sw)
    assert np.allclose(got, ref, rtol=1e-15, atol=0)


def test_w8a8_rows_exact_power_of_two_case():
    # small integers are exact e4m3 codes and power-of-two scales keep every product exact,
    # so the result is the integer dot product times 2^e (Python ints)
    rng = np.random.default_rng(32)
    a = rng.integers(-12, 13, size=(4, 128))
    w = rng.integers(-12, 13, size=(3, 128))
    sa = np.array([2.0 ** -3, 2.0 ** 2, 1.0, 2.0 ** -9], dtype=np.float32)
    got = oracle.linear_w8a8_rows_gemm(oracle.e4m3_encode(a.astype(np.float32)), sa,
                                       oracle.e4m3_encode(w.astype(np.float32)), np.float32(2.0 ** -5))
    for m in range(4):
        for n in range(3):
            dot = sum(int(a[m, k]) * int(w[n, k]) for k in range(128))
            assert got[m, n] == dot * float(sa[m]) * 2.0 ** -5


def test_w8a8_rows_matches_naive_loop():
    rng = np.random.default_rng(33)
    x = rng.standard_normal((3, 256)).astype(np.float32)
    x[1] *= 50.0
    wq = oracle.e4m3_encode(rng.standard_normal((4, 256)).astype(np.float32) * 20)
    y, xq, sa = oracle.linear_w8a8_rows(x, wq, np.float32(0.01), out_dtype="f32")
    table = oracle.e4m3_decode_table()
    for m in range(3):
        for n in range(4):
            acc = 0.0
            for k in range(256):
                acc += float(table[xq[m, k]]) * float(table[wq[n, k]])
            ref = np.float32(acc * float(sa[m]) * float(np.float32(0.01)))
            assert y[m, n] == ref
