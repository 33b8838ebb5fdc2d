"""Writes tests/golden/stack_self_drift.json: how far the float64 oracle's own stacked
prefill drifts from itself when its input moves by about one part in a million.

The stacked workload (T=2048, H=2048, 64 experts, I=768, top-8, 12 layers, seed 1) runs
free from h0 and from two perturbed copies of h0:
  * "rel_noise": every element multiplied by (1 + 2^-20 u), u uniform in [-1, 1]
    (about 1e-6 relative, a few float32 ulps);
  * "ulp_flips": one float32 ulp added to 1% of the elements, chosen at random.
For each copy the cosine of the final hidden state against the unperturbed run is recorded
at every depth, with the number of (token, slot) routing choices that differ.

The first page reports its FP8 prefill's cosine narrowing as layers are stacked ("FP8
grouped-expert prefill with on-chip int4-to-e4m3 dequant", section 3, Results).  The
reason is that a dynamically quantized layer is discontinuous in its input: a change of one
ulp in a tensor's largest element moves its scale and so every e4m3 code of the tensor.
These numbers measure that effect on the oracle alone, so that a GPU trajectory can be
held to the distance the oracle keeps from a copy of itself.

Calls only the oracle and the seeded input generators.  Run from the repository root:
    python tests/golden/make_stack_self_drift.py
(about 7 minutes on 8 cores).
"""

import json
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from workloads import stacked_inputs  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "stack_self_drift.json")
SEED = 1
DEPTH = 12


def quantized_layers(st):
    """Load-time per-tensor e4m3 quantization of each layer's v and o projections (q and k
    are dead values under identity attention)."""
    out = []
    for lw in st["layers"]:
        wv, sv = oracle.quant_act_per_tensor(lw["wv_f32"])
        wo, so = oracle.quant_act_per_tensor(lw["wo_f32"])
        out.append(dict(wv=wv, sv=sv, wo=wo, so=so, w_router=lw["w_router"],
                        w_gu=lw["w_gu"], s_gu=lw["s_gu"], w_dn=lw["w_dn"], s_dn=lw["s_dn"]))
    return out


def trajectory(h0, layers, sh):
    """Hidden state after each layer and each layer's routing ids."""
    h = np.asarray(h0, dtype=np.float32)
    states, routes = [], []
    for lw in layers:
        h, r = oracle.stacked_prefill(h, [lw], sh["k"], sh["I"], sh["n_heads"],
                                      sh["n_kv_heads"])
        states.append(h)
        routes.append(r[0])
    return states, routes


def cosine(a, b):
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    return float(a @ b / np.sqrt((a @ a) * (b @ b)))


def perturbations(h0, seed):
    rng = np.random.default_rng(seed)
    u = rng.uniform(-1.0, 1.0, h0.shape)
    rel = (h0.astype(np.float64) * (1.0 + 2.0 ** -20 * u)).astype(np.float32)
    flips = h0.copy()
    mask = rng.random(h0.shape) < 0.01
    flips[mask] = np.nextafter(flips[mask], np.float32(np.inf))
    return {"rel_noise": rel, "ulp_flips": flips}


def main():
    t0 = time.time()
    st = stacked_inputs(DEPTH, seed=SEED)
    sh = st["shape"]
    layers = quantized_layers(st)
    base, base_routes = trajectory(st["h0"], layers, sh)
    result = {
        "what": "cosine of the oracle's free-running stacked prefill from perturbed h0 "
                "against the unperturbed run, by depth",
        "workload": {"T": sh["T"], "H": sh["H"], "E": sh["E"], "I": sh["I"], "k": sh["k"],
                     "layers": DEPTH, "seed": SEED},
        "runs": {},
    }
    for name, h0p in perturbations(st["h0"], 12345).items():
        states, routes = trajectory(h0p, layers, sh)
        result["runs"][name] = {
            "input_cosine": cosine(h0p, st["h0"]),
            "cosine_by_depth": [cosine(a, b) for a, b in zip(states, base)],
            "routing_diffs_by_depth": [int(np.sum(np.sort(a, axis=1) != np.sort(b, axis=1)))
                                       for a, b in zip(routes, base_routes)],
        }
    result["seconds"] = round(time.time() - t0, 1)
    with open(OUT, "w") as f:
        json.dump(result, f, indent=1)
    print(json.dumps(result, indent=1))


if __name__ == "__main__":
    main()
