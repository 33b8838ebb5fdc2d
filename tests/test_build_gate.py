"""Build gate on the grouped GEMM's register allocation (CPU only: nvcc and ptxas, no GPU).

The int4 instances of the grouped GEMM split 128 launch registers per thread into 64 / 32 /
208 with setmaxnreg; the epilogue's 208 hold 128 fp32 accumulators, the TMEM load buffers and
the scales, and ptxas places a few spill slots there.  Asynchronous tcgen05.ld destinations
must never be spilled before their tcgen05.wait::ld (ptxas tracks them like any other
asynchronous load), and tests/test_gpu_repeat.py runs full-size GEMMs twenty times in a row
to catch any result that varies from run to run.  This gate keeps the spill space from
growing unnoticed: every instance must stay within the bytes listed below, and the e4m3
(dense and decode) instances must not spill at all."""

import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# spill-store bytes per instance <BN, bank format, epilogue>, as ptxas reports them for the
# current sources (formats: 0 LUT, 1 subnormal, 2 e4m3; epilogues: 0 f32, 1 bf16, 2 SwiGLU)
BUDGET = {
    "128/0/1": 48, "256/0/1": 24, "128/0/0": 48, "256/0/0": 48, "256/0/2": 24,
    "128/1/1": 48, "256/1/1": 24, "128/1/0": 48, "256/1/0": 48, "256/1/2": 24,
    "128/1/0/mx": 48, "128/1/1/mx": 48,
}


def _spills():
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    src = os.path.join(ROOT, "fp8_grouped_expert_gb300", "csrc", "gemm.cu")
    r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
                        "-std=c++17", "-I" + os.path.join(ROOT, "include"), "-Xptxas", "-v",
                        "-c", src, "-o", os.devnull], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    out, cur = {}, None
    for ln in r.stderr.splitlines():
        m = re.search(r"Compiling entry function '(\S+)'", ln)
        if m:
            cur = m.group(1)
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", ln)
        if m and cur and "grouped_gemm_kernel" in cur:
            g = re.search(r"ILi(\d+)ELi(\d+)ELi(\d+)ELi(\d+)E", cur).groups()
            key = "%s/%s/%s" % g[:3] + ("/mx" if g[3] == "1" else "")
            out[key] = (int(m.group(1)), int(m.group(2)))
            cur = None
    return out


@pytest.mark.skipif(not os.path.exists(os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"),
                                                    "bin", "nvcc")), reason="no nvcc")
def test_grouped_gemm_spills_stay_within_budget():
    sp = _spills()
    assert len(sp) == 18, sorted(sp)
    for key, (stores, loads) in sp.items():
        if key.split("/")[1] == "2":          # e4m3 weights: dense and decode instances
            assert stores == 0 and loads == 0, (key, stores, loads)
        else:
            assert stores <= BUDGET[key], (key, stores, BUDGET[key])


@pytest.mark.skipif(not os.path.exists(os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"),
                                                    "bin", "nvcc")), reason="no nvcc")
@pytest.mark.parametrize("src", ["decode.cu", "route.cu", "quant.cu", "glue.cu", "dispatch.cu"])
def test_other_kernels_do_not_spill(src):
    # the routing, quantization, combine, decode-projection and glue kernels keep every
    # value in registers (several hold loads in flight or bulk-copy state across waits)
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    csrc = os.path.join(ROOT, "fp8_grouped_expert_gb300", "csrc")
    r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
                        "-std=c++17", "-I" + os.path.join(ROOT, "include"), "-I" + csrc,
                        "-Xptxas", "-v", "-c", os.path.join(csrc, src), "-o", os.devnull],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    spills = re.findall(r"(\d+) bytes spill stores, (\d+) bytes spill loads", r.stderr)
    assert spills, "ptxas reported no kernels"
    assert all(s == "0" and l == "0" for s, l in spills), (src, spills)
