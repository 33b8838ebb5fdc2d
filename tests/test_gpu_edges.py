"""Edge cases of the path on the GPU: the largest expert count the grouped GEMM takes (and a
refusal one past it), a layer in which every token picks every expert (k = E, where the gates
are the plain softmax), and a layer of a single token."""

import numpy as np
import pytest
import torch

import oracle
from util import DEV, bf16_dev, cosine, host, to_dev
from workloads import moe_inputs, pack_int4

pytestmark = pytest.mark.gpu


def test_grouped_gemm_at_the_expert_limit(fge):
    # 512 experts (the limit: the kernel keeps the offsets in shared memory), rows only in
    # experts 0, 7, 255 and 511 with ragged counts, every other expert empty; small integers
    # and power-of-two scales keep the result exact
    rng = np.random.default_rng(90)
    e_count, n, k = 512, 128, 256
    counts = np.zeros(e_count, np.int64)
    counts[[0, 7, 255, 511]] = [3, 130, 1, 64]
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    r = int(offsets[-1])
    a = rng.integers(-16, 17, (r, k)).astype(np.float32)
    aq = oracle.e4m3_encode(a)
    as_ = rng.choice([1.0, 2.0], (r, k // 128)).astype(np.float32)
    q = rng.integers(-8, 8, (e_count, n, k))
    wp = pack_int4(q)
    ws = rng.choice([2.0 ** -6, 2.0 ** -5], (e_count, n, k // 128)).astype(np.float32)
    wd, sd = fge.w4_prepack(to_dev(wp), to_dev(ws))
    out = fge.grouped_gemm_w4a8(to_dev(aq), to_dev(as_), to_dev(offsets), wd, sd,
                                out_dtype=torch.float32)
    ref = oracle.grouped_gemm_w4a8(aq, as_, offsets, wp, ws)
    assert np.array_equal(host(out).astype(np.float64), ref)


def test_grouped_gemm_refuses_one_expert_past_the_limit(fge):
    e_count, n, k = 513, 128, 128
    aq = torch.zeros((4, k), dtype=torch.uint8, device=DEV)
    as_ = torch.ones((4, 1), dtype=torch.float32, device=DEV)
    offsets = torch.zeros(e_count + 1, dtype=torch.int32, device=DEV)
    wd = torch.zeros((e_count, n, k // 2), dtype=torch.uint8, device=DEV)
    sd = torch.ones((e_count, 1, n), dtype=torch.float32, device=DEV)
    with pytest.raises(fge.FgeError):
        fge.grouped_gemm_w4a8(aq, as_, offsets, wd, sd, out_dtype=torch.float32)


def _layer(fge, inp):
    w_gu, s_gu = fge.w4_prepack(to_dev(inp.w_gu), to_dev(inp.s_gu), gate_up_interleave=True)
    w_dn, s_dn = fge.w4_prepack(to_dev(inp.w_dn), to_dev(inp.s_dn))
    out = fge.moe_layer_forward(to_dev(inp.logits), bf16_dev(inp.x_bits), inp.k, inp.I, w_gu,
                                s_gu, w_dn, s_dn, out_dtype=torch.float32)
    torch.cuda.synchronize()
    return host(out)


def test_layer_with_every_expert_chosen(fge):
    inp = moe_inputs("tiny", seed=21, k=8)          # k = E = 8
    ids, gates = fge.moe_topk_gate(to_dev(inp.logits), inp.k)
    l64 = inp.logits.astype(np.float64)
    soft = np.exp(l64 - l64.max(axis=1, keepdims=True))
    soft /= soft.sum(axis=1, keepdims=True)
    ids_h, gates_h = host(ids), host(gates)
    assert np.array_equal(np.sort(ids_h, axis=1), np.tile(np.arange(8), (inp.T, 1)))
    assert np.allclose(np.take_along_axis(soft, ids_h.astype(np.int64), axis=1), gates_h,
                       rtol=2e-6, atol=0)
    got = _layer(fge, inp)
    ref, _ = oracle.moe_layer_forward(inp.logits, inp.x, inp.k, inp.w_gu, inp.s_gu, inp.w_dn,
                                      inp.s_dn, inp.I, out_dtype="f32")
    assert cosine(got, ref) >= 0.9999


def test_layer_of_one_token(fge):
    inp = moe_inputs("tiny", seed=22, T=1)
    got = _layer(fge, inp)
    ref, _ = oracle.moe_layer_forward(inp.logits, inp.x, inp.k, inp.w_gu, inp.s_gu, inp.w_dn,
                                      inp.s_dn, inp.I, out_dtype="f32")
    assert got.shape == (1, inp.H)
    assert cosine(got, ref) >= 0.9999
