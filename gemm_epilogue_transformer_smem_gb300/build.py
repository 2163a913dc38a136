"""Compiles the CUDA library (csrc/*.cu) for sm_103a into
``_build/libgemm_epi.so`` inside this package.

Each translation unit compiles in its own nvcc process, in parallel, then one
nvcc call links them.  The cudart runtime is linked statically and the
driver's tensor-map encoder is looked up at run time, so the library loads on
a machine without a GPU driver; every compute call then fails with a CUDA
error.
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
UNITS = ["gemm_epi.cu", "spec_forward.cu", "spec_aux.cu", "spec_fp8.cu", "spec_common.cu"]


def sources(csrc=CSRC):
    files = [os.path.join(csrc, f) for f in sorted(os.listdir(csrc)) if f.endswith((".cu", ".cuh"))]
    files.append(os.path.join(ROOT, "include", "gemm_epi.h"))
    return files


def compile_command(src: str, obj: str, extra=()):
    return ["nvcc", "-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC,-O2,-fvisibility=hidden",
            "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), *extra,
            "-c", "-o", obj, src]


def link_command(objs, out: str):
    return ["nvcc", *ARCH, "-shared", "-o", out, *objs]


def compile_library(csrc: str, out: str, verbose: bool = False) -> str:
    """Builds the library from the sources in `csrc` into `out`."""
    obj_dir = out + ".objs"
    os.makedirs(obj_dir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose else []
    procs, objs = [], []
    for unit in UNITS:
        obj = os.path.join(obj_dir, unit.replace(".cu", ".o"))
        objs.append(obj)
        procs.append(subprocess.Popen(compile_command(os.path.join(csrc, unit), obj, extra)))
    codes = [p.wait() for p in procs]
    if any(codes):
        raise RuntimeError("nvcc failed for %s" % [u for u, c in zip(UNITS, codes) if c])
    tmp = out + ".tmp.%d" % os.getpid()
    subprocess.run(link_command(objs, tmp), check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False, verbose: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= max(os.path.getmtime(f) for f in sources())):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    return compile_library(CSRC, LIB, verbose)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
