"""The per-token int4 dispatch baseline on the GPU against its oracle (cosine >= 0.9999),
and the source page's parity gate between the FP8 grouped path and the int4 baseline on the
same inputs (cosine >= 0.997)."""

import numpy as np
import pytest
import torch

import oracle
from util import bf16_dev, cosine, host, to_dev
from workloads import moe_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,T", [("tiny", None), ("mid", 256)])
def test_per_token_dispatch_matches_oracle_and_fp8_path(fge, name, T):
    inp = moe_inputs(name, seed=4, T=T)
    od = torch.float32 if inp.out == "f32" else torch.bfloat16
    logits, x = to_dev(inp.logits), bf16_dev(inp.x_bits)
    base = host(fge.moe_layer_per_token_dispatch(logits, x, inp.k, inp.I, to_dev(inp.w_gu),
                                                 to_dev(inp.s_gu), to_dev(inp.w_dn),
                                                 to_dev(inp.s_dn), out_dtype=od))
    ref, _ = oracle.moe_layer_int4_baseline(inp.logits, inp.x, inp.k, inp.w_gu, inp.s_gu,
                                            inp.w_dn, inp.s_dn, inp.I, out_dtype=inp.out)
    assert cosine(base, ref) >= 0.9999
    w_gu, s_gu = fge.w4_prepack(to_dev(inp.w_gu), to_dev(inp.s_gu), True)
    w_dn, s_dn = fge.w4_prepack(to_dev(inp.w_dn), to_dev(inp.s_dn), False)
    fp8 = host(fge.moe_layer_forward(logits, x, inp.k, inp.I, w_gu, s_gu, w_dn, s_dn,
                                     out_dtype=od))
    c = cosine(fp8, base)
    print("FP8 grouped path vs int4 per-token baseline, cosine %.6f" % c)
    assert c >= 0.997
