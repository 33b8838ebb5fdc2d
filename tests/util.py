"""Helpers shared by the GPU parity tests: host <-> device conversion and the tolerance
checks of the parity rules (bit-exact integers/codes; GEMMs normwise <= 2e-3 and
elementwise |d| <= 1 bf16 ulp(ref) + 1e-5 * sum|as*sw*a*w|; layers cosine >= 0.9999)."""

import numpy as np
import torch

import oracle

DEV = torch.device("cuda:0")


def bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(DEV)


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def host(t):
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy()
    return t.cpu().numpy()


def bf16_ulp(ref):
    a = np.abs(np.asarray(ref, dtype=np.float64))
    _, e = np.frexp(np.maximum(a, 2.0 ** -126))
    return np.ldexp(1.0, e - 1 - 7)


def abs_grouped(aq, as_, offsets, w_packed, w_scale):
    """sum_g |as*sw| * sum_k |a| |q| per output (the elementwise error scale)."""
    a = np.abs(oracle.e4m3_decode(aq))
    r, kdim = a.shape
    e_count, n, _ = w_packed.shape
    g = kdim // 128
    out = np.zeros((r, n))
    for e in range(e_count):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r0 == r1:
            continue
        w = np.abs(oracle.int4_unpack(w_packed[e], kdim).astype(np.float64))
        for gi in range(g):
            ks = slice(gi * 128, gi * 128 + 128)
            out[r0:r1] += (np.abs(as_[r0:r1, gi:gi + 1].astype(np.float64))
                           * np.abs(w_scale[e, :, gi].astype(np.float64))[None, :]
                           * (a[r0:r1, ks] @ w[:, ks].T))
    return out


def check_gemm(got, ref, absref, bf16_out):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    norm = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    assert norm <= 2e-3, "normwise relative error %.3e" % norm
    tol = 1e-5 * absref + (bf16_ulp(ref) if bf16_out else 1e-6 * np.abs(ref))
    bad = np.abs(got - ref) > tol
    assert not bad.any(), "elementwise bound violated at %d places, worst %s" % (
        bad.sum(), np.max(np.abs(got - ref) - tol))
    return norm


def cosine(a, b):
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    return float(a @ b / np.sqrt((a @ a) * (b @ b)))
