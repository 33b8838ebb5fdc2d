"""The oracle's pins must catch plausible mistakes.

Each case below plants one mistake in the numpy oracle (on the CPU, through monkeypatch, for
the duration of the test only): a dropped term, a wrong sign or index, a swapped operand, a
rounding or tie rule changed.  It then runs the pins that should see it and requires at
least one of them to fail.  A pin set that let one of these through would not be tying the
oracle to the pages.
"""

import numpy as np
import pytest

import oracle
import oracle.fp8 as ofp8
import oracle.moe as omoe
import oracle.mx as omx
import test_oracle_fp8 as pf
import test_oracle_moe as pm
import test_oracle_mx_gemm as pmx

_NAMESPACES = (oracle, ofp8, omoe)


def _patch(monkeypatch, name, fn):
    for ns in _NAMESPACES:
        if hasattr(ns, name):
            monkeypatch.setattr(ns, name, fn)


def _must_fail(*pins):
    failed = 0
    for pin in pins:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed > 0, "no pin caught the planted mistake"


# --- codec ------------------------------------------------------------------------------------

def _encode_with(round_fn, saturate=True):
    table = ofp8.e4m3_decode_table()
    pos = table[0:0x7F]

    def enc(x):
        x64 = np.asarray(x, dtype=np.float32).astype(np.float64)
        neg = np.signbit(x64)
        a = np.abs(np.where(np.isinf(x64), 1e9, x64))
        _, e = np.frexp(a)
        quantum = np.ldexp(1.0, np.maximum(e - 1, -6) - 3)
        q = round_fn(a / quantum) * quantum
        if saturate:
            q = np.minimum(q, 448.0)
        code = np.searchsorted(pos, np.minimum(q, 448.0))
        code = np.where(q > 448.0, 0x7F, code)
        return (code.astype(np.uint8) | (neg.astype(np.uint8) << 7)).astype(np.uint8)
    return enc


def test_ties_away_from_zero_is_caught(monkeypatch):
    _patch(monkeypatch, "e4m3_encode", _encode_with(lambda v: np.floor(v + 0.5)))
    _must_fail(pf.test_encode_ties_go_to_even_code, pf.test_encode_subnormal_rounding)


def test_truncation_is_caught(monkeypatch):
    _patch(monkeypatch, "e4m3_encode", _encode_with(np.floor))
    _must_fail(pf.test_encode_matches_torch_cast_in_range, pf.test_quant_closed_form_group)


def test_missing_saturation_is_caught(monkeypatch):
    _patch(monkeypatch, "e4m3_encode", _encode_with(np.rint, saturate=False))
    _must_fail(pf.test_encode_saturates_and_keeps_sign)


def test_high_nibble_first_is_caught(monkeypatch):
    def unpack(packed, k):
        p = np.asarray(packed, dtype=np.uint8)
        lo, hi = (p >> 4).astype(np.int16), (p & 0x0F).astype(np.int16)
        out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.int8)
        out[..., 0::2] = np.where(lo >= 8, lo - 16, lo)
        out[..., 1::2] = np.where(hi >= 8, hi - 16, hi)
        return out
    _patch(monkeypatch, "int4_unpack", unpack)
    _must_fail(pf.test_int4_nibble_order_and_sign)
    _must_fail(pm.test_grouped_gemm_matches_naive_loop_on_tiny_case)


def test_missing_sign_extension_is_caught(monkeypatch):
    def unpack(packed, k):
        p = np.asarray(packed, dtype=np.uint8)
        out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.int8)
        out[..., 0::2] = p & 0x0F
        out[..., 1::2] = p >> 4
        return out
    _patch(monkeypatch, "int4_unpack", unpack)
    _must_fail(pf.test_int4_nibble_order_and_sign)
    _must_fail(pm.test_grouped_gemm_exact_small_integer_case)


def test_bf16_double_rounding_is_caught(monkeypatch):
    orig = ofp8.bf16_round
    _patch(monkeypatch, "bf16_round",
           lambda x: orig(np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)))
    _must_fail(pf.test_bf16_round_single_rounding_from_float64)


# --- quantization ---------------------------------------------------------------------------

def test_wrong_divisor_is_caught(monkeypatch):
    # 240, the largest finite value of the e4m3 variant without NaN/inf reuse, instead of 448
    orig = ofp8._scale_from_amax
    monkeypatch.setattr(ofp8, "_scale_from_amax", lambda a: orig(a) * np.float32(448 / 240))
    _must_fail(pf.test_quant_closed_form_group, pf.test_quant_error_bound)


def test_missing_zero_floor_is_caught(monkeypatch):
    def scale(amax):
        with np.errstate(divide="ignore", invalid="ignore"):
            return (np.asarray(amax, dtype=np.float32) / np.float32(448.0)).astype(np.float32)
    monkeypatch.setattr(ofp8, "_scale_from_amax", scale)
    with np.errstate(divide="ignore", invalid="ignore"):
        _must_fail(pf.test_quant_zero_group_gives_zero_codes_and_unit_scale,
                   pf.test_quant_tiny_group_scale_floor)


def test_multiplying_by_the_scale_is_caught(monkeypatch):
    def quant(x_f32):
        x = np.asarray(x_f32, dtype=np.float32)
        m, k = x.shape
        g = x.reshape(m, k // 128, 128)
        s = ofp8._scale_from_amax(np.max(np.abs(g), axis=2))
        return ofp8.e4m3_encode(g * s[:, :, None]).reshape(m, k), s
    _patch(monkeypatch, "quant_act_g128", quant)
    _must_fail(pf.test_quant_closed_form_group)


# --- routing, permutation ------------------------------------------------------------------

def test_ties_to_the_higher_expert_are_caught(monkeypatch):
    def topk(logits, k):
        lg = np.asarray(logits, dtype=np.float32)
        t, e = lg.shape
        ids = np.empty((t, k), np.int32)
        gates = np.empty((t, k), np.float32)
        for row in range(t):
            order = sorted(range(e), key=lambda j: (-float(lg[row, j]), -j))[:k]
            w = np.exp(np.array([float(lg[row, j]) for j in order]) - float(lg[row, order[0]]))
            ids[row], gates[row] = order, w / w.sum()
        return ids, gates
    _patch(monkeypatch, "topk_gate", topk)
    _must_fail(pm.test_topk_ties_choose_lower_ids_and_equal_gates)


def test_unrenormalised_gates_are_caught(monkeypatch):
    orig = omoe.topk_gate

    def topk(logits, k):
        ids, _ = orig(logits, k)
        lg = np.asarray(logits, dtype=np.float64)
        full = np.exp(lg - lg.max(1, keepdims=True))
        full /= full.sum(1, keepdims=True)
        return ids, np.take_along_axis(full, ids.astype(np.int64), 1).astype(np.float32)
    _patch(monkeypatch, "topk_gate", topk)
    _must_fail(pm.test_topk_gates_renormalise_full_softmax)


def test_unstable_permutation_is_caught(monkeypatch):
    orig = omoe.moe_permute

    def permute(ids, num_experts, xq, xs):
        # same counts and offsets, tokens reversed inside every expert
        p = orig(ids, num_experts, xq, xs)
        rt = p["row_token"].copy()
        for e in range(num_experts):
            a, b = p["offsets"][e], p["offsets"][e + 1]
            rt[a:b] = rt[a:b][::-1]
        p["row_token"] = rt
        p["aq"] = np.asarray(xq)[rt]
        p["as_"] = np.asarray(xs)[rt]
        return p
    _patch(monkeypatch, "moe_permute", permute)
    _must_fail(pm.test_permute_invariants)


# --- GEMMs, SwiGLU, combine ----------------------------------------------------------------

def _gemm_variant(kind):
    def gemm(aq, as_, offsets, w_packed, w_scale):
        aq = np.asarray(aq)
        r_total, kdim = aq.shape
        e_count, n, _ = np.asarray(w_packed).shape
        a = ofp8.e4m3_decode(aq)
        out = np.zeros((r_total, n))
        for e in range(e_count):
            r0, r1 = int(offsets[e]), int(offsets[e + 1])
            if r1 == r0:
                continue
            w = ofp8.int4_unpack(w_packed[e], kdim).astype(np.float64)
            for g in range(kdim // 128):
                ks = slice(g * 128, (g + 1) * 128)
                part = a[r0:r1, ks] @ w[:, ks].T
                sa = np.asarray(as_[r0:r1, g], dtype=np.float64)[:, None]
                sw = np.asarray(w_scale[e, :, 0 if kind == "group0" else g], np.float64)[None, :]
                if kind == "no_act_scale":
                    sa = np.ones_like(sa)
                out[r0:r1] += sa * sw * part
        return out
    return gemm


@pytest.mark.parametrize("kind", ["group0", "no_act_scale"])
def test_grouped_gemm_scale_mistakes_are_caught(monkeypatch, kind):
    _patch(monkeypatch, "grouped_gemm_w4a8", _gemm_variant(kind))
    _must_fail(pm.test_grouped_gemm_exact_small_integer_case,
               pm.test_grouped_gemm_all_ones_closed_form)


def test_wrong_expert_weights_are_caught(monkeypatch):
    orig = omoe.grouped_gemm_w4a8

    def gemm(aq, as_, offsets, w_packed, w_scale):
        return orig(aq, as_, offsets, np.roll(w_packed, 1, axis=0), np.roll(w_scale, 1, axis=0))
    _patch(monkeypatch, "grouped_gemm_w4a8", gemm)
    _must_fail(pm.test_grouped_gemm_exact_small_integer_case)


def test_gate_up_halves_swapped_are_caught(monkeypatch):
    orig = omoe.swiglu_requant

    def swiglu(c, inter):
        c = np.asarray(c, dtype=np.float64)
        return orig(np.concatenate([c[:, inter:2 * inter], c[:, :inter]], axis=1), inter)
    _patch(monkeypatch, "swiglu_requant", swiglu)
    _must_fail(pm.test_swiglu_closed_forms_and_library_silu)


def test_combine_ignoring_gates_is_caught(monkeypatch):
    orig = omoe.moe_combine
    _patch(monkeypatch, "moe_combine",
           lambda y, token_row, gates: orig(y, token_row, np.ones_like(gates)))
    _must_fail(pm.test_combine_linear_in_gates)


def test_w8a8_missing_weight_scale_is_caught(monkeypatch):
    orig = omoe.linear_w8a8_gemm
    _patch(monkeypatch, "linear_w8a8_gemm", lambda aq, sa, wq, sw: orig(aq, sa, wq, 1.0))
    _must_fail(pm.test_w8a8_exact_power_of_two_case)


# --- MXFP4-activation grouped GEMM ---------------------------------------------------------------

def _mx_dequant_with(block):
    """mx_dequant_e2m1 that applies the scale of the wrong block: k // block instead of k // 32
    (block 16: twice as many scales read; block 128: one scale per group)."""
    def deq(packed, scales):
        packed = np.asarray(packed, dtype=np.uint8)
        scales = np.asarray(scales, dtype=np.uint8)
        m, kh = packed.shape
        table = np.array([omx.e2m1_decode(c) for c in range(16)])
        out = np.empty((m, 2 * kh), dtype=np.float64)
        out[:, 0::2] = table[packed & 0xF]
        out[:, 1::2] = table[packed >> 4]
        idx = np.minimum(np.arange(2 * kh) // block, scales.shape[1] - 1)
        return out * 2.0 ** (scales[:, idx].astype(np.float64) - 127.0)
    return deq


@pytest.mark.parametrize("block", [16, 128])
def test_mx_gemm_wrong_scale_block_is_caught(monkeypatch, block):
    monkeypatch.setattr(omx, "mx_dequant_e2m1", _mx_dequant_with(block))
    _must_fail(pmx.test_block_scale_placement_closed_form,
               pmx.test_equals_w4a8_when_block_scales_agree_within_groups)


def test_mx_gemm_wrong_scale_bias_is_caught(monkeypatch):
    real = omx.mx_dequant_e2m1
    monkeypatch.setattr(omx, "mx_dequant_e2m1", lambda p, s: real(p, s) * 2.0)   # bias 126
    _must_fail(pmx.test_block_scale_placement_closed_form,
               pmx.test_equals_w4a8_when_block_scales_agree_within_groups)
