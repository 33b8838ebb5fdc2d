"""In-tree build of libfge.so (the C-ABI CUDA library) for sm_103a.

Each translation unit under csrc/ is compiled by nvcc in parallel, then linked into
fp8_grouped_expert_gb300/libfge.so.  A rebuild happens only when a source or header is newer
than the library.  No cmake; plain nvcc, one -gencode.
"""

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfge.so")
SOURCES = ["api.cu", "quant.cu", "route.cu", "gemm.cu", "glue.cu", "noalloc.cu", "selftest.cu", "dispatch.cu",
           "decode.cu"]
HEADERS = ["fge_device.cuh", "fge_internal.h", os.path.join("..", "..", "include", "fge.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I" + os.path.join(ROOT, "include")]


def nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale(sources, target):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in sources)


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed: %s\n%s%s" % (" ".join(cmd), r.stdout, r.stderr))
    return r.stdout + r.stderr


def build(verbose=False, ptxas_info=False):
    """Compile and link libfge.so if anything changed; returns the library path."""
    os.makedirs(BUILD, exist_ok=True)
    headers = [os.path.join(CSRC, h) for h in HEADERS]
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    if not _stale(srcs + headers + [__file__], LIB) and not ptxas_info:
        return LIB
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src).replace(".cu", ".o"))
        if ptxas_info or _stale([src] + headers + [__file__], obj):
            out = _run([nvcc()] + NVCC_FLAGS + extra + ["-c", src, "-o", obj])
            if verbose or ptxas_info:
                sys.stdout.write(out)
        return obj

    with ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = LIB + ".tmp"
    _run([nvcc()] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="--ptxas" in sys.argv))
