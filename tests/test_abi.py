"""The C-ABI library builds, loads and exports every entry point that include/fge.h
declares, and the Python binding declares a signature for each.  No compute calls."""

import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "fge.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fge_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def mod():
    from fp8_grouped_expert_gb300 import build as _build
    _build.build()
    import fp8_grouped_expert_gb300 as m
    m.lib()
    return m


def test_header_declares_the_hot_path_calls():
    names = _declared()
    for needed in ["fge_fp8_quant_act", "fge_moe_topk_gate", "fge_moe_permute",
                   "fge_grouped_gemm_w4a8", "fge_swiglu_quant", "fge_moe_combine",
                   "fge_gemm_w8a8", "fge_linear_w8a8", "fge_moe_layer_forward",
                   "fge_w4_prepack", "fge_init", "fge_workspace_bytes"]:
        assert needed in names


def test_library_exports_every_declared_symbol(mod):
    lib = mod.lib()
    for name in _declared():
        assert hasattr(lib, name), name
        assert name in mod.SIGNATURES, "binding lacks a signature for " + name


def test_host_only_queries(mod):
    lib = mod.lib()
    assert lib.fge_version() >= 100
    assert mod.status_string(0) == "ok"
    assert "workspace" in mod.status_string(4)
    assert mod.workspace_bytes(mod.OP_GROUPED_GEMM) == 256
    lay = mod.workspace_bytes(mod.OP_MOE_LAYER, 4096, 2048, 768, 64, 8)
    # at least the permuted activations, the SwiGLU output and the expert outputs
    assert lay > 32768 * 2048 + 32768 * 768 + 32768 * 2048 * 2
    assert mod.workspace_bytes(mod.OP_LINEAR_W8A8, 16, 2560) >= 256 + 16 * 2560
    assert mod.workspace_bytes(99) == 0


def test_calls_without_init_or_with_bad_args_fail_before_launch(mod):
    lib = mod.lib()
    # no device has been initialised in this CPU process, so every compute entry point
    # refuses before touching the GPU
    st = lib.fge_moe_topk_gate(None, 0, 8, 2, None, None, None)
    assert st != 0
    assert lib.fge_init(-1) == 1  # invalid argument


def test_ledger_counts_refusals_without_a_gpu(mod):
    lib = mod.lib()
    mod.reset_ledger()
    assert mod.ledger() == {k: 0 for k in ("calls", "refused", "layers", "grouped_gemms",
                                           "dense_decode_tile", "dense_row_tile")}
    # three compute calls on a process with no initialised device: all refused before launch
    assert lib.fge_moe_topk_gate(None, 0, 8, 2, None, None, None) != 0
    assert lib.fge_moe_combine(None, 0, None, None, 0, 1, 128, 0, None, None) != 0
    assert lib.fge_rmsnorm(None, 0, 128, 1e-6, None, None) != 0
    led = mod.ledger()
    assert led["calls"] == 3 and led["refused"] == 3 and led["layers"] == 0
    mod.reset_ledger()
    assert mod.ledger()["calls"] == 0


def test_status_strings_cover_the_device_codes(mod):
    assert "timed out" in mod.status_string(mod.ERR_DEVICE_TIMEOUT)
    assert "NaN" in mod.status_string(mod.ERR_NONFINITE)
