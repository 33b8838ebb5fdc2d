"""A plain C program (tests/c_abi/linear_closed_form.c) calls the library through
include/fge.h with device memory from the CUDA runtime -- no Python and no PyTorch between
it and the ABI.  On the CPU it must compile against the header; on the GPU it is linked with
libfge.so and run, and checks a closed form of fge_linear_w8a8 at a decode size and at a
128-row size, a refused NULL pointer and the status strings."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "linear_closed_form.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")
GCC = shutil.which("gcc")


def _flags():
    return ["-std=c11", "-O1", "-Wall", "-Werror", "-I" + os.path.join(ROOT, "include"),
            "-I" + os.path.join(CUDA, "include")]


@pytest.mark.skipif(GCC is None, reason="no gcc")
def test_c_caller_compiles_against_the_header(tmp_path):
    r = subprocess.run([GCC] + _flags() + ["-c", SRC, "-o", str(tmp_path / "c.o")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


@pytest.mark.gpu
def test_c_caller_runs_on_the_gpu(fge, tmp_path):
    lib_dir = os.path.dirname(fge.lib()._name)
    exe = tmp_path / "linear_closed_form"
    r = subprocess.run([GCC] + _flags() + [SRC, "-o", str(exe), "-L" + lib_dir, "-lfge",
                        "-L" + os.path.join(CUDA, "lib64"), "-lcudart",
                        "-Wl,-rpath," + lib_dir, "-Wl,-rpath," + os.path.join(CUDA, "lib64")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "c_abi ok" in run.stdout
