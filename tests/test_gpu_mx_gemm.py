"""GPU parity of the grouped GEMM with MXFP4 activations (fge_grouped_gemm_mxf4_w4: E2M1
codes with one power-of-two scale per 32 values, applied inside tcgen05 block-scaled MMAs)
against the oracle's definition, oracle.grouped_gemm_mxf4_w4.

Exact cases first, where every product, every K = 32 step and the fp32 accumulation are
exact, so the kernel must reproduce the oracle bit for bit:
  * one scale for everything (checks the MMA kind, the padded E2M1 operand and the int4
    side);
  * scales that differ per row and per 32-value block within +-1 binade (checks where each
    scale sits in TMEM: a row or K step read from the wrong place changes a power of two);
then quantized bf16 activations (the library's own MXFP4 quantizer, bit-exact to the oracle
elsewhere) on routed, ragged row sets under the elementwise GEMM rule."""

import numpy as np
import pytest
import torch

import oracle
from util import bf16_ulp, cosine, host, to_dev
from workloads import pack_int4

pytestmark = pytest.mark.gpu


def _pack_codes(codes):
    codes = np.asarray(codes, dtype=np.uint8)
    return np.ascontiguousarray((codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8))


def _bank(fge, q, sw):
    return fge.w4_prepack(to_dev(pack_int4(q)), to_dev(sw), fmt=fge.W4_SUBNORMAL)


def _run(fge, packed, scales, offsets, q, sw, out_dtype=torch.float32):
    wd, sd = _bank(fge, q, sw)
    ws = fge.new_workspace(fge.workspace_bytes(fge.OP_GROUPED_GEMM), wd.device)
    fge.clear_device_status(ws)
    out = fge.grouped_gemm_mxf4_w4(to_dev(packed), to_dev(scales), to_dev(offsets), wd, sd,
                                   out_dtype=out_dtype, workspace=ws)
    assert fge.read_device_status(ws) == 0
    return host(out)


def _exact_case(rng, counts, n, k, scale_fn):
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    r = int(offsets[-1])
    codes = rng.integers(0, 16, (r, k)).astype(np.uint8)
    scales = scale_fn(r, k).astype(np.uint8)
    q = rng.integers(-8, 8, (len(counts), n, k))
    sw = rng.choice([2.0 ** -6, 2.0 ** -5], (len(counts), n, k // 128)).astype(np.float32)
    return _pack_codes(codes), scales, offsets, q, sw


def test_mx_gemm_refusals(fge):
    dev = torch.device("cuda:0")
    codes = torch.zeros((128, 64), dtype=torch.uint8, device=dev)
    scales = torch.zeros((128, 4), dtype=torch.uint8, device=dev)
    offsets = torch.tensor([0, 128], dtype=torch.int32, device=dev)
    q = np.zeros((1, 128, 128), dtype=np.int64)
    wd, sd = _bank(fge, q, np.ones((1, 128, 1), np.float32))
    with pytest.raises(fge.FgeError):       # K/32 scales per row required
        fge.grouped_gemm_mxf4_w4(codes, scales[:, :2], offsets, wd, sd)
    misaligned = torch.zeros(128 * 64 + 16, dtype=torch.uint8, device=dev)[16:].view(128, 64)
    with pytest.raises(fge.FgeError):       # the padded-E2M1 copy wants a 32-byte base
        fge.grouped_gemm_mxf4_w4(misaligned, scales, offsets, wd, sd)


def test_mx_gemm_exact_one_scale(fge):
    rng = np.random.default_rng(41)
    packed, scales, offsets, q, sw = _exact_case(
        rng, [128], 128, 128, lambda r, k: np.full((r, k // 32), 128))
    got = _run(fge, packed, scales, offsets, q, sw)
    ref = oracle.grouped_gemm_mxf4_w4(packed, scales, offsets, pack_int4(q), sw)
    assert np.array_equal(got.astype(np.float64), ref)


@pytest.mark.parametrize("counts,n,k", [([128], 128, 128), ([130, 0, 70, 1], 256, 384)])
def test_mx_gemm_exact_scales_per_row_and_block(fge, counts, n, k):
    rng = np.random.default_rng(43 + k)
    packed, scales, offsets, q, sw = _exact_case(
        rng, counts, n, k, lambda r, kk: rng.integers(126, 129, (r, kk // 32)))
    got = _run(fge, packed, scales, offsets, q, sw)
    ref = oracle.grouped_gemm_mxf4_w4(packed, scales, offsets, pack_int4(q), sw)
    assert np.array_equal(got.astype(np.float64), ref)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("t,e,kk,h,n", [(97, 8, 2, 512, 256), (300, 16, 4, 1024, 384)])
def test_mx_gemm_quantized_activations(fge, out_dtype, t, e, kk, h, n):
    rng = np.random.default_rng(t + n)
    lg = (rng.standard_normal((t, e)) - 1.1 * np.log(np.arange(1, e + 1))).astype(np.float32)
    ids, _ = oracle.topk_gate(lg, kk)
    x = rng.standard_normal((t, h)).astype(np.float32)
    x[:, rng.choice(h, 8, replace=False)] *= 20.0
    xb = torch.from_numpy(x).to(torch.bfloat16)
    codes_t, scales_t = oracle.mx_quant_e2m1(xb.float().numpy().astype(np.float64))
    # routed rows in expert order: row r of the grouped GEMM is token row_token[r]
    perm = oracle.moe_permute(ids, e, np.zeros((t, h), np.uint8), np.zeros((t, h // 128),
                                                                          np.float32))
    rt = perm["row_token"]
    packed, scales = np.ascontiguousarray(codes_t[rt]), np.ascontiguousarray(scales_t[rt])
    q = rng.integers(-8, 8, (e, n, h))
    sw = rng.uniform(0.002, 0.02, (e, n, h // 128)).astype(np.float32)
    got = _run(fge, packed, scales, perm["offsets"], q, sw, out_dtype).astype(np.float64)
    ref = oracle.grouped_gemm_mxf4_w4(packed, scales, perm["offsets"], pack_int4(q), sw)
    # elementwise: 1 bf16 ulp of the result (bf16 output) plus 1e-5 of sum |sw * a * q|
    a_abs = np.abs(oracle.mx_dequant_e2m1(packed, scales))
    absref = np.zeros_like(ref)
    offs = perm["offsets"]
    for ei in range(e):
        r0, r1 = int(offs[ei]), int(offs[ei + 1])
        if r1 > r0:
            wabs = np.abs(q[ei].astype(np.float64)) * np.repeat(sw[ei].astype(np.float64), 128,
                                                                  axis=1)
            absref[r0:r1] = a_abs[r0:r1] @ wabs.T
    tol = 1e-5 * absref + (bf16_ulp(ref) if out_dtype == torch.bfloat16 else 1e-6 * np.abs(ref))
    assert np.all(np.abs(got - ref) <= tol), np.max(np.abs(got - ref) - tol)
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 2e-3
    assert cosine(got, ref) > 0.99999
