"""Compile the CUDA sources into the in-tree shared library libmlora.so.

nvcc, one -gencode for sm_103a, no fast-math (IEEE division and no
flush-to-zero), translation units compiled in parallel, then linked with the
static CUDA runtime.  The library needs no other CUDA library at run time
(the tensor-map encoder is fetched from the driver through the runtime).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmlora.so")
SOURCES = ("api.cu", "plan.cu", "shrink.cu", "shrink_mma.cu", "gemm.cu", "gemm_sk.cu", "accept.cu", "softmax.cu", "kvcache.cu", "fp8.cu", "noalloc.cu")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmlora.so")


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
                   "-I" + os.path.join(ROOT, "include"), *extra]


def build(verbose: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile every translation unit and link libmlora.so.  Returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []

    def one(src):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [cc, *_flags(extra), "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        outs = list(ex.map(one, SOURCES))
    if verbose or ptxas_verbose:
        for _, log in outs:
            if log.strip():
                print(log)
    tmp = LIB + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *[o for o, _ in outs], "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(verbose=True, ptxas_verbose="-v" in sys.argv))
