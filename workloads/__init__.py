"""Seeded synthetic inputs for the MoE prefill path and the dense W8A8 projection.

These generators are the only code that the CUDA path's tests and the CPU oracle share.
They hold none of the method's arithmetic: they draw random numbers, round them to bf16
(a storage format), pack int4 values two per byte (the weight bank's storage format, low
nibble = even k) and, for the stacked workload, build int4 weights from Gaussian draws with
a per-group absmax/7 rule that is weight preparation, not part of the prefill path.  The
e4m3 weights of the dense projections are NOT produced here: each side quantizes the bf16
weights with its own per-tensor quantizer, at load.

Workloads (sizes and distributions of the MoE prefill and dense-projection cases):
  tiny    T=64,    H=256,  E=8,   I=512,  top-2, fp32 output
  dense   N=6656,  K=2560, M in {16, 256, 2048, 8192}, bf16 output
  mid     T=4096,  H=2048, E=64,  I=768,  top-8, bf16 output
  large   T=16384, H=4096, E=128, I=1536, top-8, Zipf(1.1) router bias, 1% outlier channels
  stacked T=2048,  H=2048, L layers of dense q/k/v/o (16 q heads, 4 kv heads of 128) + MoE
"""

import zlib
from dataclasses import dataclass, field

import numpy as np
import torch

GROUP = 128

MOE_SHAPES = {
    "tiny": dict(T=64, H=256, E=8, I=512, k=2, out="f32"),
    "mid": dict(T=4096, H=2048, E=64, I=768, k=8, out="bf16"),
    "large": dict(T=16384, H=4096, E=128, I=1536, k=8, out="bf16"),
}
DENSE_SHAPE = dict(N=6656, K=2560, Ms=(16, 256, 2048, 8192))
STACK_SHAPE = dict(T=2048, H=2048, E=64, I=768, k=8, n_heads=16, n_kv_heads=4, q=2048,
                   kv=512)


def _seq(*parts):
    words = []
    for p in parts:
        words.append(zlib.crc32(p.encode()) if isinstance(p, str) else int(p))
    return np.random.SeedSequence(words)


def to_bf16(x_f32):
    """float32 array -> (uint16 bf16 bits, float32 values of those bf16), round to nearest."""
    t = torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32)).to(torch.bfloat16)
    bits = t.view(torch.int16).numpy().view(np.uint16).copy()
    return bits, t.float().numpy()


def pack_int4(q):
    """int values in -8..7, shape [..., K] -> uint8 [..., K/2]; element 2b in the low nibble."""
    q = np.asarray(q, dtype=np.int16)
    if q.size and (q.min() < -8 or q.max() > 7):
        raise ValueError("int4 values must lie in -8..7")
    nib = (q & 0xF).astype(np.uint8)
    return (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)


@dataclass
class MoEInputs:
    name: str
    T: int
    H: int
    E: int
    I: int
    k: int
    out: str
    x_bits: np.ndarray        # uint16 [T, H]  bf16 activations
    x: np.ndarray             # float32 [T, H] values of x_bits
    logits: np.ndarray        # float32 [T, E]
    w_gu: np.ndarray          # uint8 [E, 2I, H/2] packed int4 (rows 0..I-1 gate, I..2I-1 up)
    s_gu: np.ndarray          # float32 [E, 2I, H/128]
    w_dn: np.ndarray          # uint8 [E, H, I/2]
    s_dn: np.ndarray          # float32 [E, H, I/128]
    meta: dict = field(default_factory=dict)


def _uniform_int4_bank(rng, e, n, k):
    q = rng.integers(-8, 8, size=(e, n, k), dtype=np.int8)
    return pack_int4(q)


def _uniform_scales(rng, e, n, k):
    return rng.uniform(0.002, 0.02, size=(e, n, k // GROUP)).astype(np.float32)


def moe_inputs(name, seed=0, T=None, **overrides):
    """Inputs of one MoE layer.  ``T`` (and H, E, I, k) override the shape; the
    distributions stay those of the named workload."""
    sh = dict(MOE_SHAPES[name])
    if T is not None:
        sh["T"] = T
    sh.update(overrides)
    t, h, e, inter, k = sh["T"], sh["H"], sh["E"], sh["I"], sh["k"]
    rng = np.random.default_rng(_seq(seed, "moe", name, t, h, e, inter, k))
    x = rng.standard_normal((t, h), dtype=np.float32)
    logits = rng.standard_normal((t, e), dtype=np.float32)
    meta = {}
    if name == "large":
        # per-expert router bias = log of the unnormalised Zipf(1.1) pmf of rank e+1
        bias = (-1.1 * np.log(np.arange(1, e + 1, dtype=np.float64))).astype(np.float32)
        logits = (logits + bias[None, :]).astype(np.float32)
        n_out = int(0.01 * h)
        chans = rng.choice(h, size=n_out, replace=False)
        x[:, chans] *= np.float32(20.0)
        meta["outlier_channels"] = np.sort(chans)
    x_bits, x_vals = to_bf16(x)
    w_gu = _uniform_int4_bank(rng, e, 2 * inter, h)
    s_gu = _uniform_scales(rng, e, 2 * inter, h)
    w_dn = _uniform_int4_bank(rng, e, h, inter)
    s_dn = _uniform_scales(rng, e, h, inter)
    return MoEInputs(name, t, h, e, inter, k, sh["out"], x_bits, x_vals, logits, w_gu, s_gu,
                     w_dn, s_dn, meta)


@dataclass
class DenseInputs:
    M: int
    N: int
    K: int
    x_bits: np.ndarray   # uint16 [M, K]
    x: np.ndarray        # float32 [M, K]
    w_bits: np.ndarray   # uint16 [N, K] bf16 weights, quantized per tensor at load by each side
    w: np.ndarray        # float32 [N, K]


def dense_weight(seed=0, N=None, K=None):
    """bf16 projection weight ~N(0, 0.02), [N, K]."""
    n = N or DENSE_SHAPE["N"]
    kk = K or DENSE_SHAPE["K"]
    rng = np.random.default_rng(_seq(seed, "dense_w", n, kk))
    w = (rng.standard_normal((n, kk), dtype=np.float32) * np.float32(0.02)).astype(np.float32)
    return to_bf16(w)


def dense_activations(m, k, seed=0):
    """bf16 activations ~N(0, 1), [M, K]."""
    rng = np.random.default_rng(_seq(seed, "dense_x", m, k))
    return to_bf16(rng.standard_normal((m, k), dtype=np.float32))


def dense_activations_outliers(m, k, seed=0, frac=0.01, factor=20.0):
    """bf16 activations ~N(0, 1), [M, K], with floor(frac * K) seeded channels (columns)
    multiplied by `factor` (the outlier-channel recipe of the large skewed MoE workload)."""
    rng = np.random.default_rng(_seq(seed, "dense_x_outliers", m, k))
    x = rng.standard_normal((m, k), dtype=np.float32)
    cols = rng.choice(k, size=int(frac * k), replace=False)
    x[:, cols] *= np.float32(factor)
    return to_bf16(x)


def dense_activations_outlier_rows(m, k, seed=0, frac=0.01, factor=20.0):
    """bf16 activations ~N(0, 1), [M, K], with max(1, floor(frac * M)) seeded rows (tokens)
    multiplied by `factor`."""
    rng = np.random.default_rng(_seq(seed, "dense_x_outlier_rows", m, k))
    x = rng.standard_normal((m, k), dtype=np.float32)
    rows = rng.choice(m, size=max(1, int(frac * m)), replace=False)
    x[rows] *= np.float32(factor)
    return to_bf16(x)


def dense_inputs(M, seed=0, N=None, K=None):
    n = N or DENSE_SHAPE["N"]
    kk = K or DENSE_SHAPE["K"]
    w_bits, w = dense_weight(seed, n, kk)
    x_bits, x = dense_activations(M, kk, seed)
    return DenseInputs(M, n, kk, x_bits, x, w_bits, w)


def _int4_from_gaussian(rng, e, n, k, std):
    """Weight preparation for the stacked workload: w ~ N(0, std); per (row, 128 group)
    s = absmax/7 (float32); q = clamp(round_half_even(w/s), -8, 7)."""
    w = (rng.standard_normal((e, n, k), dtype=np.float32) * np.float32(std)).astype(np.float32)
    g = w.reshape(e, n, k // GROUP, GROUP)
    amax = np.max(np.abs(g), axis=3)
    s = (amax / np.float32(7.0)).astype(np.float32)
    s = np.where(s == 0, np.float32(1.0), s).astype(np.float32)
    q = np.clip(np.rint(g / s[..., None]), -8, 7).astype(np.int8).reshape(e, n, k)
    return pack_int4(q), s


def stacked_inputs(L, seed=0, T=None):
    """Inputs of an L-layer stack: h0 ~ N(0,1) float32; per layer bf16 dense weights
    ~N(0,0.02) for q [2048x2048], k/v [512x2048], o [2048x2048]; router fp32 ~N(0,0.02)
    [E x H]; int4 expert banks built from N(0,0.02) draws."""
    sh = dict(STACK_SHAPE)
    if T is not None:
        sh["T"] = T
    t, h, e, inter = sh["T"], sh["H"], sh["E"], sh["I"]
    rng = np.random.default_rng(_seq(seed, "stack", L, t))
    h0 = rng.standard_normal((t, h), dtype=np.float32)
    layers = []
    for _ in range(L):
        lw = {}
        for name, rows in (("q", sh["q"]), ("k", sh["kv"]), ("v", sh["kv"]), ("o", h)):
            w = (rng.standard_normal((rows, h), dtype=np.float32) * np.float32(0.02))
            lw["w" + name + "_bits"], lw["w" + name + "_f32"] = to_bf16(w)
        lw["w_router"] = (rng.standard_normal((e, h), dtype=np.float32)
                          * np.float32(0.02)).astype(np.float32)
        lw["w_gu"], lw["s_gu"] = _int4_from_gaussian(rng, e, 2 * inter, h, 0.02)
        lw["w_dn"], lw["s_dn"] = _int4_from_gaussian(rng, e, h, inter, 0.02)
        layers.append(lw)
    return dict(shape=sh, L=L, h0=h0, layers=layers)
