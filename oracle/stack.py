"""Oracle: stacked prefill layers (RMSNorm, dense W8A8 q/k/v/o, identity attention, router,
MoE FFN, float32 residual).

Test infrastructure only (see the package docstring).  The composition is pinned by two
properties (zero weights give the identity; token permutations commute with the stack) and
each piece by its own pins; the GPU stack is compared with it by cosine similarity of the
final hidden state and by the count of routing choices that differ, as the source page
compares its FP8 prefill by logit cosine ("FP8 grouped-expert prefill with on-chip
int4-to-e4m3 dequant", sections 1 and 3).
"""

import numpy as np

from .fp8 import bf16_bits_to_f32, bf16_round
from .moe import linear_w8a8, moe_layer_forward

RMS_EPS = 1e-6
HEAD_DIM = 128


def rmsnorm(h):
    """x / sqrt(mean(x^2) + 1e-6) per row with unit gain, float64, rounded to bf16.

    Not on the pages; reading: a pre-norm block with unit gain and eps 1e-6.
    """
    h64 = np.asarray(h, dtype=np.float64)
    r = h64 / np.sqrt(np.mean(h64 * h64, axis=1, keepdims=True) + RMS_EPS)
    return bf16_bits_to_f32(bf16_round(r))


def router_logits(xn, w_router):
    """Router logits = xn @ Wr^T, float64 dot products rounded to float32."""
    return (np.asarray(xn, dtype=np.float64)
            @ np.asarray(w_router, dtype=np.float64).T).astype(np.float32)


def identity_attention(v, n_heads, n_kv_heads):
    """Attention core replaced by identity on v, with grouped-query head sharing.

    Reading: query head h reads kv head h // (n_heads / n_kv_heads), so
    attn[t, h*128 + d] = v[t, (h // rep)*128 + d].
    """
    v = np.asarray(v)
    rep = n_heads // n_kv_heads
    t = v.shape[0]
    heads = v.reshape(t, n_kv_heads, HEAD_DIM)
    return np.repeat(heads, rep, axis=1).reshape(t, n_heads * HEAD_DIM)


def stacked_prefill(h0, layers, k, inter, n_heads, n_kv_heads):
    """Run L layers; each layer dict holds wv/sv, wo/so (e4m3 codes + fp32 scale),
    w_router (fp32 [E, H]) and the MoE banks w_gu/s_gu, w_dn/s_dn.

    Per layer: xn = RMSNorm(h); v = W8A8(xn, Wv) (q and k are dead values under identity
    attention and are not needed for the result); attn = identity(v); h += W8A8(attn, Wo);
    xn2 = RMSNorm(h); logits = xn2 Wr^T; h += MoE(xn2).  h stays float32.
    Returns (h float32 [T, H], list of per-layer routing ids).
    """
    h = np.asarray(h0, dtype=np.float32).copy()
    routes = []
    for lw in layers:
        xn = rmsnorm(h)
        v, _, _ = linear_w8a8(xn, lw["wv"], lw["sv"])
        attn = identity_attention(v, n_heads, n_kv_heads)
        o, _, _ = linear_w8a8(attn, lw["wo"], lw["so"])
        h = (h.astype(np.float64) + o.astype(np.float64)).astype(np.float32)
        xn2 = rmsnorm(h)
        logits = router_logits(xn2, lw["w_router"])
        y, inter_d = moe_layer_forward(logits, xn2, k, lw["w_gu"], lw["s_gu"], lw["w_dn"],
                                       lw["s_dn"], inter, out_dtype="bf16")
        routes.append(inter_d["ids"])
        h = (h.astype(np.float64) + y.astype(np.float64)).astype(np.float32)
    return h, routes
