"""Compiles the CUDA library (csrc/gemm_epi.cu) for sm_103a into
``_build/libgemm_epi.so`` inside this package.

The cudart runtime is linked statically and the driver's tensor-map encoder is
looked up at run time, so the library loads on a machine without a GPU
driver; every compute call then fails with a CUDA error.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libgemm_epi.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def sources():
    files = [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC))
             if f.endswith((".cu", ".cuh"))]
    files.append(os.path.join(ROOT, "include", "gemm_epi.h"))
    return files


def nvcc_command(out: str, extra=()):
    return (["nvcc", "-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC,-O2",
             "-shared", "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"),
             *extra, "-o", out, os.path.join(CSRC, "gemm_epi.cu")])


def build(force: bool = False, verbose: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= max(os.path.getmtime(f) for f in sources())):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = nvcc_command(tmp, ["-Xptxas", "-v"] if verbose else [])
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
