"""Oracle: routing, permutation, grouped W4A8 GEMM, SwiGLU requant, combine, dense W8A8.

Test infrastructure only (see the package docstring).  Everything is float64 unless a step
is defined in float32.
"""

import numpy as np

from .fp8 import (
    bf16_round,
    bf16_bits_to_f32,
    e4m3_decode,
    int4_unpack,
    quant_act_g128,
    quant_act_per_row,
    quant_act_per_tensor,
)

GROUP = 128


def topk_gate(logits, k):
    """Top-k expert choice per token with softmax gates over the chosen logits.

    The pages only say that routed tokens are dispatched to experts ("FP8 grouped-expert
    prefill with on-chip int4-to-e4m3 dequant", section 1).  Reading (standard top-k MoE
    routing): order the E logits of a token descending, ties broken toward the lower expert
    id; keep the first k; gate_j = exp(l_j - l_max) / sum over the k chosen of
    exp(l - l_max), which equals the full softmax renormalised over the chosen experts.

    logits: float32 [T, E].  Returns (ids int32 [T, k], gates float32 [T, k]).
    """
    lg = np.asarray(logits, dtype=np.float32)
    t, e = lg.shape
    if not 1 <= k <= e:
        raise ValueError("need 1 <= k <= E")
    ids = np.empty((t, k), dtype=np.int32)
    gates = np.empty((t, k), dtype=np.float32)
    for row in range(t):
        order = sorted(range(e), key=lambda j: (-float(lg[row, j]), j))[:k]
        chosen = np.array([float(lg[row, j]) for j in order], dtype=np.float64)
        w = np.exp(chosen - chosen.max())
        ids[row] = order
        gates[row] = (w / w.sum()).astype(np.float32)
    return ids, gates


def moe_permute(ids, num_experts, xq, xs):
    """Group routed (token, slot) pairs into expert-contiguous rows.

    Replaces one dispatch per routed token with one grouped GEMM over all of them ("FP8
    grouped-expert prefill with on-chip int4-to-e4m3 dequant", section 1), which needs the
    routed rows of each expert to be contiguous.  Steps: counts[e] = number of pairs routed
    to e; offsets = exclusive prefix sum of counts; rows are ordered by (expert, token
    ascending, slot ascending) -- a stable counting sort; row r copies the quantized
    activation row and its group scales from token row_token[r].

    ids: int [T, k]; xq: uint8 [T, H]; xs: float32 [T, H/128].
    Returns dict(counts, offsets [E+1], row_token [R], token_row [T, k], aq [R, H],
    as_ [R, H/128]) with R = T*k, all integer outputs int32.
    """
    ids = np.asarray(ids, dtype=np.int64)
    t, k = ids.shape
    counts = np.zeros(num_experts, dtype=np.int64)
    for e in ids.ravel():
        counts[e] += 1
    offsets = np.zeros(num_experts + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    cursor = offsets[:-1].copy()
    row_token = np.empty(t * k, dtype=np.int64)
    token_row = np.empty((t, k), dtype=np.int64)
    for tok in range(t):
        for j in range(k):
            e = ids[tok, j]
            r = cursor[e]
            cursor[e] += 1
            row_token[r] = tok
            token_row[tok, j] = r
    return dict(
        counts=counts.astype(np.int32),
        offsets=offsets.astype(np.int32),
        row_token=row_token.astype(np.int32),
        token_row=token_row.astype(np.int32),
        aq=np.asarray(xq)[row_token],
        as_=np.asarray(xs, dtype=np.float32)[row_token],
    )


def grouped_gemm_w4a8(aq, as_, offsets, w_packed, w_scale):
    """One grouped expert GEMM over all routed rows, int4 weights, e4m3 activations.

    "FP8 grouped-expert prefill with on-chip int4-to-e4m3 dequant", section 1: a single
    grouped expert GEMM per layer; int4 weights dequantized to e4m3 without unpacking the
    resident bank; a per-(token, group) activation scale folded into the accumulator path.
    Definition written out: for expert e and its rows r in [offsets[e], offsets[e+1]),
        C[r, n] = sum_g  as[r, g] * sw[e, n, g] * sum_{k in group g} dec(aq[r, k]) * q[e, n, k]
    with q the int4 values (exact in e4m3, so the on-chip dequant changes nothing).  Each
    inner group sum is exact in float64 (products have at most 7 significant bits and there
    are 128 terms); scaling and the outer sum are float64.

    aq uint8 [R, K]; as_ float32 [R, K/128]; offsets int [E+1]; w_packed uint8 [E, N, K/2];
    w_scale float32 [E, N, K/128].  Returns float64 [R, N] (rows past offsets[E] are zero).
    """
    aq = np.asarray(aq)
    r_total, kdim = aq.shape
    e_count, n, _ = np.asarray(w_packed).shape
    groups = kdim // GROUP
    a = e4m3_decode(aq)
    out = np.zeros((r_total, n), dtype=np.float64)
    for e in range(e_count):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            continue
        w = int4_unpack(w_packed[e], kdim).astype(np.float64)
        acc = np.zeros((r1 - r0, n), dtype=np.float64)
        for g in range(groups):
            ks = slice(g * GROUP, (g + 1) * GROUP)
            partial = a[r0:r1, ks] @ w[:, ks].T
            scale = (np.asarray(as_[r0:r1, g], dtype=np.float64)[:, None]
                     * np.asarray(w_scale[e, :, g], dtype=np.float64)[None, :])
            acc += scale * partial
        out[r0:r1] = acc
    return out


def linear_w8a8_gemm(aq, sa, wq, sw):
    """Dense per-tensor W8A8 GEMM: Y = (sa * sw) * dec(Aq) @ dec(Wq)^T in float64.

    "feat(qwen4_exp): load-time per-tensor FP8 dense projections", section "What this adds"
    (e4m3 weights with one fp32 scale, dynamic per-tensor activation scale) and "Module
    fp8_ffi" (activation scale folded with the weight scale into one scalar applied to the
    GEMM).  The grouped kernel run with one group computes the same thing.
    """
    a = e4m3_decode(aq)
    w = e4m3_decode(wq)
    return (float(np.float32(sa)) * float(np.float32(sw))) * (a @ w.T)


def swiglu_requant(c, inter):
    """SwiGLU between the two expert GEMMs, then e4m3 requant per (row, 128 group).

    Not described on the pages (the expert FFN is named, not its activation).  Reading: the
    merged gate_up output holds gate in columns [0, I) and up in [I, 2I); the accumulator is
    float32 on the device, so C is first rounded to float32; h = fp32(silu(g) * u) with
    silu(g) = g / (1 + exp(-g)) evaluated in float64; then the activation quantization of
    ``quant_act_g128`` runs over h.  Returns (hq uint8 [R, I], hs float32 [R, I/128], h).
    """
    c32 = np.asarray(c, dtype=np.float64).astype(np.float32).astype(np.float64)
    g = c32[:, :inter]
    u = c32[:, inter:2 * inter]
    h = (g / (1.0 + np.exp(-g)) * u).astype(np.float32)
    hq, hs = quant_act_g128(h)
    return hq, hs, h


def moe_combine(y, token_row, gates):
    """Gate-weighted sum of each token's k expert rows back into token order.

    Reading (the pages do not describe it): out[t] = sum over slots j = 0..k-1, in slot
    order, of gates[t, j] * y[token_row[t, j]], accumulated in float64.
    y: float [R, N]; token_row int [T, k]; gates float32 [T, k].  Returns float64 [T, N].
    """
    y = np.asarray(y, dtype=np.float64)
    token_row = np.asarray(token_row)
    gates = np.asarray(gates, dtype=np.float32).astype(np.float64)
    t, k = token_row.shape
    out = np.zeros((t, y.shape[1]), dtype=np.float64)
    for j in range(k):
        out += gates[:, j:j + 1] * y[token_row[:, j]]
    return out


def _round_out(v, out_dtype):
    if out_dtype == "f32":
        return np.asarray(v, dtype=np.float64).astype(np.float32)
    return bf16_bits_to_f32(bf16_round(v))


def moe_layer_forward(logits, x_f32, k, w_gate_up, s_gate_up, w_down, s_down, inter,
                      out_dtype="bf16"):
    """One MoE FFN prefill layer: quant -> route -> permute -> gate_up -> SwiGLU requant ->
    down -> combine.

    Follows the stage order of the grouped-expert prefill ("FP8 grouped-expert prefill with
    on-chip int4-to-e4m3 dequant", section 1) with the readings of the functions above.
    The expert outputs y are stored in ``out_dtype`` (bf16 or f32) before the combine, as
    they leave the down GEMM; the combine output is rounded to ``out_dtype``.
    Returns (out float32 values [T, H], intermediates dict).
    """
    ids, gates = topk_gate(logits, k)
    xq, xs = quant_act_g128(x_f32)
    num_experts = np.asarray(w_gate_up).shape[0]
    perm = moe_permute(ids, num_experts, xq, xs)
    c = grouped_gemm_w4a8(perm["aq"], perm["as_"], perm["offsets"], w_gate_up, s_gate_up)
    hq, hs, h = swiglu_requant(c, inter)
    y = grouped_gemm_w4a8(hq, hs, perm["offsets"], w_down, s_down)
    y_st = _round_out(y, out_dtype)
    out = _round_out(moe_combine(y_st, perm["token_row"], gates), out_dtype)
    inter_d = dict(ids=ids, gates=gates, xq=xq, xs=xs, c=c, hq=hq, hs=hs, h=h, y=y_st, **perm)
    return out, inter_d


def linear_w8a8(x_f32, wq, sw, out_dtype="bf16"):
    """Dense projection: dynamic per-tensor activation quant, then the W8A8 GEMM, rounded
    to ``out_dtype``.  Returns (y float32 values [M, N], xq, sa)."""
    xq, sa = quant_act_per_tensor(x_f32)
    y = linear_w8a8_gemm(xq, sa, wq, sw)
    return _round_out(y, out_dtype), xq, sa


def dequant_int4_bank(w_packed, w_scale, k):
    """Dequantized expert bank in float64: W[e, n, kk] = q[e, n, kk] * sw[e, n, kk // 128]."""
    q = int4_unpack(w_packed, k).astype(np.float64)
    s = np.repeat(np.asarray(w_scale, dtype=np.float64), GROUP, axis=-1)
    return q * s


def moe_layer_int4_baseline(logits, x_f32, k, w_gate_up, s_gate_up, w_down, s_down, inter,
                            out_dtype="bf16"):
    """The per-token int4 expert dispatch that the grouped GEMM replaces ("FP8 grouped-expert
    prefill with on-chip int4-to-e4m3 dequant", section 1: its baseline runs one dispatch per
    routed token with the int4 weights).  Reading: activations are not quantized; for each
    routed (token, slot) the expert FFN is y = W_down (silu(W_gate x) * (W_up x)) with the
    dequantized int4 weights, in float64; out[t] = sum_j gate_j * y_j, rounded to out_dtype.
    Returns (out float32 values [T, H], ids)."""
    ids, gates = topk_gate(logits, k)
    x = np.asarray(x_f32, dtype=np.float64)
    t_count, h = x.shape
    out = np.zeros((t_count, h), dtype=np.float64)
    for e in np.unique(ids):
        tok, slot = np.nonzero(ids == e)
        wgu = dequant_int4_bank(w_gate_up[e:e + 1], s_gate_up[e:e + 1], h)[0]
        wdn = dequant_int4_bank(w_down[e:e + 1], s_down[e:e + 1], inter)[0]
        c = x[tok] @ wgu.T
        g, u = c[:, :inter], c[:, inter:2 * inter]
        y = (g / (1.0 + np.exp(-g)) * u) @ wdn.T
        out[tok] += gates[tok, slot].astype(np.float64)[:, None] * y
    return _round_out(out, out_dtype), ids


def linear_w8a8_rows_gemm(aq, sa_rows, wq, sw):
    """Dense W8A8 GEMM with one activation scale per row: Y[m, n] = (sa[m] * sw) *
    sum_k dec(Aq[m, k]) * dec(Wq[n, k]), in float64 ("feat(qwen4_exp) ...", section
    "Limits": row-wise activation scales instead of the per-tensor one)."""
    a = e4m3_decode(aq)
    w = e4m3_decode(wq)
    scale = np.asarray(sa_rows, dtype=np.float32).astype(np.float64) * float(np.float32(sw))
    return scale[:, None] * (a @ w.T)


def linear_w8a8_rows(x_f32, wq, sw, out_dtype="bf16"):
    """Dense projection with row-wise activation scales: per-row quantization, then
    ``linear_w8a8_rows_gemm``, rounded to ``out_dtype``.  Returns (y, xq, sa [M])."""
    xq, sa = quant_act_per_row(x_f32)
    y = linear_w8a8_rows_gemm(xq, sa, wq, sw)
    return _round_out(y, out_dtype), xq, sa
