"""The oracle's own sensitivity in the stacked prefill (T=2048, 12 layers): the committed
fixture tests/golden/stack_self_drift.json, written by tests/golden/make_stack_self_drift.py
from the oracle alone, holds the cosine of the oracle's free-running final state from an input
moved by about 1e-6 (relative noise 2^-20, and separately one float32 ulp on 1% of the
elements) against the unperturbed run, at every depth.

Why it matters: a layer that quantizes its activations dynamically (per-tensor and per-group
e4m3 scales from the data's amax) is discontinuous in its input, so any two implementations
that round differently in the last bits (fp32 on the GPU, float64 here) drift apart with depth
exactly as a perturbed copy of one implementation does ("FP8 grouped-expert prefill with
on-chip int4-to-e4m3 dequant", section 3, Results, reports its own cosine narrowing with
depth).  The GPU free-running test is held to these numbers."""

import json
import os

import numpy as np

import oracle
from workloads import pack_int4

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FIXTURE = os.path.join(ROOT, "tests", "golden", "stack_self_drift.json")


def _fixture():
    with open(FIXTURE) as f:
        return json.load(f)


def test_fixture_describes_the_stacked_workload():
    d = _fixture()
    assert d["workload"] == {"T": 2048, "H": 2048, "E": 64, "I": 768, "k": 8, "layers": 12,
                             "seed": 1}
    for run in ("rel_noise", "ulp_flips"):
        r = d["runs"][run]
        assert len(r["cosine_by_depth"]) == 12 and len(r["routing_diffs_by_depth"]) == 12
        assert r["input_cosine"] > 1 - 1e-12


def test_oracle_drifts_from_itself_with_depth():
    r = _fixture()["runs"]["rel_noise"]
    c = np.array(r["cosine_by_depth"])
    # the drift grows with depth (every step down, allowing no rise beyond 1e-7)
    assert np.all(np.diff(c) < 1e-7)
    assert c[0] > 0.99999 and c[3] < 0.99999 and c[11] < 0.9995
    # routing choices that differ grow with it (near-tie flips after a scale moved)
    d = np.array(r["routing_diffs_by_depth"])
    assert d[11] > d[3] > d[0] >= 0
    # the values the GPU bound is built from (depth 4, 8, 12)
    assert abs(c[3] - 0.99995618) < 1e-7
    assert abs(c[7] - 0.99953675) < 1e-7
    assert abs(c[11] - 0.99905968) < 1e-7


def test_smaller_perturbation_drifts_less():
    runs = _fixture()["runs"]
    flips = np.array(runs["ulp_flips"]["cosine_by_depth"])
    noise = np.array(runs["rel_noise"]["cosine_by_depth"])
    assert np.all(1 - flips <= 1 - noise + 1e-12)


def test_the_mechanism_on_a_small_stack():
    """The same effect on a small stack (seconds on the CPU): moving the input by one part in
    a million leaves the first layer almost exact and then the states drift apart, because a
    changed amax moves a whole tensor's e4m3 codes."""
    rng = np.random.default_rng(3)
    H, E, I, T, L = 256, 8, 256, 256, 6
    layers = []
    for _ in range(L):
        wv, sv = oracle.quant_act_per_tensor((rng.standard_normal((128, H)) * 0.05).astype(np.float32))
        wo, so = oracle.quant_act_per_tensor((rng.standard_normal((H, 256)) * 0.05).astype(np.float32))
        layers.append(dict(wv=wv, sv=sv, wo=wo, so=so,
                           w_router=(rng.standard_normal((E, H)) * 0.05).astype(np.float32),
                           w_gu=pack_int4(rng.integers(-8, 8, (E, 2 * I, H))),
                           s_gu=rng.uniform(5e-4, 2e-3, (E, 2 * I, H // 128)).astype(np.float32),
                           w_dn=pack_int4(rng.integers(-8, 8, (E, H, I))),
                           s_dn=rng.uniform(5e-4, 2e-3, (E, H, I // 128)).astype(np.float32)))
    h0 = rng.standard_normal((T, H)).astype(np.float32)
    h0p = (h0.astype(np.float64) * (1 + 2.0 ** -20 * rng.uniform(-1, 1, h0.shape))).astype(np.float32)
    a, b = h0, h0p
    cos = []
    for lw in layers:
        a, _ = oracle.stacked_prefill(a, [lw], 2, I, 2, 1)
        b, _ = oracle.stacked_prefill(b, [lw], 2, I, 2, 1)
        a64, b64 = a.astype(np.float64).ravel(), b.astype(np.float64).ravel()
        cos.append(a64 @ b64 / np.sqrt((a64 @ a64) * (b64 @ b64)))
    assert cos[0] > 1 - 1e-5
    assert cos[-1] < cos[0]                   # drifted with depth
    assert not np.array_equal(a, b)
