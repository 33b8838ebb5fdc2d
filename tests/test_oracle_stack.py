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
