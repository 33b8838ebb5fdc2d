"""Pins for the stacked prefill's composition (the layer pieces have their own pins).

Two properties fix it beyond its pieces: with every projection and expert weight zero the
stack is the identity on the hidden state (each block adds exactly zero to the residual),
and it is equivariant under a permutation of the tokens (every step acts per token, and the
per-tensor scales are taken over the whole tensor, which a permutation does not change).
A dropped or replaced residual, rows mixed up anywhere, or a norm over the wrong axis fails
one of these or the pieces' own pins; the planted versions below check that they do."""

import numpy as np
import pytest

import oracle
import oracle.stack as ostack
from workloads import pack_int4


def _layers(rng, n, H=256, E=8, I=256, nkv=1, nh=2, zero=False):
    layers = []
    for _ in range(n):
        wv = np.zeros((nkv * 128, H), np.float32) if zero else \
            (rng.standard_normal((nkv * 128, H)) * 0.02).astype(np.float32)
        wo = np.zeros((H, nh * 128), np.float32) if zero else \
            (rng.standard_normal((H, nh * 128)) * 0.02).astype(np.float32)
        wvq, sv = oracle.quant_act_per_tensor(wv)
        woq, so = oracle.quant_act_per_tensor(wo)
        q_gu = np.zeros((E, 2 * I, H), np.int8) if zero else rng.integers(-8, 8, (E, 2 * I, H))
        q_dn = np.zeros((E, H, I), np.int8) if zero else rng.integers(-8, 8, (E, H, I))
        layers.append(dict(
            wv=wvq, sv=sv, wo=woq, so=so,
            w_router=(rng.standard_normal((E, H)) * 0.02).astype(np.float32),
            w_gu=pack_int4(q_gu), s_gu=rng.uniform(5e-4, 2e-3, (E, 2 * I, H // 128)).astype(np.float32),
            w_dn=pack_int4(q_dn), s_dn=rng.uniform(5e-4, 2e-3, (E, H, I // 128)).astype(np.float32)))
    return layers


def _identity_pin():
    rng = np.random.default_rng(31)
    h0 = rng.standard_normal((20, 256)).astype(np.float32)
    h, routes = oracle.stacked_prefill(h0, _layers(rng, 3, zero=True), 2, 256, 2, 1)
    assert np.array_equal(h, h0)
    assert len(routes) == 3 and all(r.shape == (20, 2) for r in routes)


def _equivariance_pin():
    rng = np.random.default_rng(32)
    layers = _layers(rng, 2)
    h0 = rng.standard_normal((24, 256)).astype(np.float32)
    perm = rng.permutation(24)
    h, routes = oracle.stacked_prefill(h0, layers, 2, 256, 2, 1)
    hp, routes_p = oracle.stacked_prefill(h0[perm], layers, 2, 256, 2, 1)
    assert np.array_equal(hp, h[perm])
    assert all(np.array_equal(rp, r[perm]) for r, rp in zip(routes, routes_p))
    assert not np.array_equal(h, h0)                      # the stack did change h


def test_zero_weights_give_the_identity():
    _identity_pin()


def test_token_permutation_equivariance():
    _equivariance_pin()


def test_planted_norm_over_the_wrong_axis_is_caught(monkeypatch):
    def bad_rmsnorm(h):
        h64 = np.asarray(h, dtype=np.float64)
        r = h64 / np.sqrt(np.mean(h64 * h64, axis=0, keepdims=True) + 1e-6)
        return oracle.bf16_bits_to_f32(oracle.bf16_round(r))
    monkeypatch.setattr(ostack, "rmsnorm", bad_rmsnorm)
    monkeypatch.setattr(oracle, "rmsnorm", bad_rmsnorm)
    # a norm over the token axis is itself permutation-equivariant, so the composition pins
    # pass; the RMSNorm piece's closed form (rows of different scale) catches it
    import test_oracle_moe as pm
    with pytest.raises(AssertionError):
        pm.test_rmsnorm_closed_form_and_identity_attention()


def test_planted_replaced_residual_is_caught(monkeypatch):
    # a block that overwrites the residual instead of adding to it
    def bad_stack(h0, layers, k, inter, n_heads, n_kv_heads):
        h = np.asarray(h0, dtype=np.float32).copy()
        for lw in layers:
            xn = ostack.rmsnorm(h)
            v, _, _ = ostack.linear_w8a8(xn, lw["wv"], lw["sv"])
            o, _, _ = ostack.linear_w8a8(ostack.identity_attention(v, n_heads, n_kv_heads),
                                         lw["wo"], lw["so"])
            h = o.astype(np.float32)                      # residual dropped
            xn2 = ostack.rmsnorm(h)
            y, _ = ostack.moe_layer_forward(ostack.router_logits(xn2, lw["w_router"]), xn2, k,
                                            lw["w_gu"], lw["s_gu"], lw["w_dn"], lw["s_dn"],
                                            inter, out_dtype="bf16")
            h = (h.astype(np.float64) + y.astype(np.float64)).astype(np.float32)
        return h, []
    monkeypatch.setattr(oracle, "stacked_prefill", bad_stack)
    with pytest.raises(AssertionError):
        _identity_pin()


# ---------------------------------------------------------------------------------------
# Layer order.  The pins above cannot tell the two norms of a layer apart (with zero
# projections the residual does not move, so both norms see the same rows).  These build a
# layer whose attention half has a closed form: rows h = c_t * sign with c_t a power of two
# normalise to exactly the signs in bf16; v and o projections that copy channels (e4m3
# weight 1.0, per-tensor scale 1/448 on both operands) reproduce their input exactly; the
# grouped-query repeat then gives attn[t, j] = sign[t, j mod 128].  So after the attention
# residual h1 = h + sign[:, j mod 128] exactly, and h1 is not a multiple of h: a router or
# MoE that reads the first norm's output instead of the second's gives a different layer.

def _order_layer(rng, H=256, E=8, I=256, zero_moe=False):
    wv = np.zeros((128, H), np.float32)
    wv[np.arange(128), np.arange(128)] = 1.0        # v copies channels 0..127
    wo = np.eye(H, dtype=np.float32)                 # o copies its input
    wvq, sv = oracle.quant_act_per_tensor(wv)
    woq, so = oracle.quant_act_per_tensor(wo)
    q_gu = np.zeros((E, 2 * I, H), np.int8) if zero_moe else rng.integers(-8, 8, (E, 2 * I, H))
    q_dn = np.zeros((E, H, I), np.int8) if zero_moe else rng.integers(-8, 8, (E, H, I))
    return dict(wv=wvq, sv=sv, wo=woq, so=so,
                w_router=(rng.standard_normal((E, H)) * 0.5).astype(np.float32),
                w_gu=pack_int4(q_gu),
                s_gu=rng.uniform(5e-4, 2e-3, (E, 2 * I, H // 128)).astype(np.float32),
                w_dn=pack_int4(q_dn),
                s_dn=rng.uniform(5e-4, 2e-3, (E, H, I // 128)).astype(np.float32))


def _order_rows(rng, T=32, H=256):
    sign = np.where(rng.random((T, H)) < 0.5, -1.0, 1.0).astype(np.float32)
    c = (2.0 ** rng.integers(-1, 3, (T, 1))).astype(np.float32)
    return (c * sign).astype(np.float32), sign


def _attention_half_pin():
    rng = np.random.default_rng(41)
    h, sign = _order_rows(rng)
    h1 = h + sign[:, np.arange(256) % 128]               # closed form of the attention half
    out, _ = oracle.stacked_prefill(h, [_order_layer(rng, zero_moe=True)], 2, 256, 2, 1)
    assert np.array_equal(out, h1)                       # zero experts add exactly zero


def _moe_half_pin():
    rng = np.random.default_rng(42)
    h, sign = _order_rows(rng)
    lw = _order_layer(rng)
    h1 = h + sign[:, np.arange(256) % 128]
    xn2 = oracle.rmsnorm(h1)                             # the second norm reads h1
    y, _ = oracle.moe_layer_forward(oracle.router_logits(xn2, lw["w_router"]), xn2, 2,
                                    lw["w_gu"], lw["s_gu"], lw["w_dn"], lw["s_dn"], 256,
                                    out_dtype="bf16")
    want = (h1.astype(np.float64) + y.astype(np.float64)).astype(np.float32)
    out, _ = oracle.stacked_prefill(h, [lw], 2, 256, 2, 1)
    assert not np.array_equal(want, h1)                  # the experts did contribute
    assert np.array_equal(out, want)


def test_attention_half_closed_form():
    _attention_half_pin()


def test_moe_reads_the_second_norm():
    _moe_half_pin()


def _planted_stack(router_from_first_norm=False, moe_from_first_norm=False,
                   attention_on_raw=False):
    def stack(h0, layers, k, inter, n_heads, n_kv_heads):
        h = np.asarray(h0, dtype=np.float32).copy()
        for lw in layers:
            xn = ostack.rmsnorm(h)
            v, _, _ = ostack.linear_w8a8(h if attention_on_raw else xn, lw["wv"], lw["sv"])
            o, _, _ = ostack.linear_w8a8(ostack.identity_attention(v, n_heads, n_kv_heads),
                                         lw["wo"], lw["so"])
            h = (h.astype(np.float64) + o.astype(np.float64)).astype(np.float32)
            xn2 = ostack.rmsnorm(h)
            lg = ostack.router_logits(xn if router_from_first_norm else xn2, lw["w_router"])
            y, _ = ostack.moe_layer_forward(lg, xn if moe_from_first_norm else xn2, k,
                                            lw["w_gu"], lw["s_gu"], lw["w_dn"], lw["s_dn"],
                                            inter, out_dtype="bf16")
            h = (h.astype(np.float64) + y.astype(np.float64)).astype(np.float32)
        return h, []
    return stack


@pytest.mark.parametrize("mistake", ["router_from_first_norm", "moe_from_first_norm"])
def test_planted_first_norm_reader_is_caught(monkeypatch, mistake):
    monkeypatch.setattr(oracle, "stacked_prefill", _planted_stack(**{mistake: True}))
    with pytest.raises(AssertionError):
        _moe_half_pin()


def test_planted_attention_on_unnormed_rows_is_caught(monkeypatch):
    monkeypatch.setattr(oracle, "stacked_prefill", _planted_stack(attention_on_raw=True))
    with pytest.raises(AssertionError):
        _attention_half_pin()


def test_unplanted_stack_passes_the_order_pins(monkeypatch):
    # the restated stack used for the planted versions is itself correct: with no mistake
    # planted it passes both pins (so the failures above come from the planted mistakes)
    monkeypatch.setattr(oracle, "stacked_prefill", _planted_stack())
    _attention_half_pin()
    _moe_half_pin()
