"""CPU oracle for the W4A8 grouped-expert MoE prefill path and the dense W8A8 projection.

TEST INFRASTRUCTURE ONLY. Nothing in the product library imports, links or calls this
package: only the test suite, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it.

What it is: a plain, slow, float64 restatement of what the method computes, written from
the source pages ("FP8 grouped-expert prefill with on-chip int4-to-e4m3 dequant" and its
companion pages on per-tensor FP8 projections, the ``fp8_ffi`` prefill module and the FP8
vs INT4 comparison).  Each function cites the passage it follows and lists the reading it
takes where the pages are silent.  numpy matmul is the only library primitive used for a
contraction; every quantization, rounding and ordering rule is written out here.

Two restatements live here, written separately and sharing no code: this numpy package
(float64, numpy matmul as the one library primitive for a contraction) and a plain,
single-threaded C++ one (``oracle_ref.cpp``, bound by ``oracle.native`` through ctypes and
compiled with g++ by ``oracle.native.build()``) whose layer call is also the timed CPU
baseline.  Where a rule can be written two ways they take different routes, and the tests
hold them to each other as well as to the pins below.

Neither shares code with the CUDA path (``fp8_grouped_expert_gb300``): oracle and library meet only in
the seeded input generators of ``workloads``, which hold none of the method's arithmetic.

Pins (tests marked ``not gpu``) tie each function to facts the pages and the mathematics
fix: the e4m3 code table, int4 exactness in e4m3, exact power-of-two GEMMs, closed forms,
brute force on tiny inputs, and the permutation invariants; the stacked prefill's
composition by its zero-weight identity and token-permutation equivariance.  A function
whose result were only checked by a similarity measure would say "parity unpinned" in its
docstring; none is left.
"""

from .fp8 import (  # noqa: F401
    E4M3_MAX,
    e4m3_decode_table,
    e4m3_decode,
    e4m3_encode,
    int4_unpack,
    bf16_round,
    bf16_bits_to_f32,
    quant_act_g128,
    quant_act_per_tensor,
    quant_act_per_row,
)
from .mx import (  # noqa: F401
    E2M1_MAX,
    MX_BLOCK,
    e2m1_decode,
    e2m1_encode,
    mx_block_exponent,
    mx_quant_e2m1,
    mx_dequant_e2m1,
    grouped_gemm_mxf4_w4,
)
from .moe import (  # noqa: F401
    topk_gate,
    moe_permute,
    grouped_gemm_w4a8,
    linear_w8a8_gemm,
    swiglu_requant,
    moe_combine,
    moe_layer_forward,
    linear_w8a8,
    dequant_int4_bank,
    moe_layer_int4_baseline,
    linear_w8a8_rows_gemm,
    linear_w8a8_rows,
)
from .stack import rmsnorm, router_logits, identity_attention, stacked_prefill  # noqa: F401
