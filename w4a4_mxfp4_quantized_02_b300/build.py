"""Build the CUDA library ``libmacaq.so`` in-tree for sm_103a (B300).

Each translation unit is compiled with nvcc for ``compute_103a``/``sm_103a``
only; the units with transform arithmetic (the quantisation kernels and the
GEMM, whose epilogue can encode MXFP4) additionally with ``-fmad=false`` (their
arithmetic must not be contracted into FMAs).  The CUDA runtime is linked
statically and the driver API is reached through the runtime's entry-point
query, so the library loads on machines without a GPU driver (for symbol and
argument checks) and needs no JIT cache at run time.  It links no other
library: every kernel is the library's own.
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmacaq.so")
INCLUDE = os.path.join(ROOT, "include")

NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]
UNITS = {
    "quant.cu": ["-fmad=false"],
    "gemm.cu": ["-fmad=false"],
    "api.cu": [],
    "static_scratch.cu": [],
    "flip.cu": ["-fmad=false"],
    "moe.cu": ["-fmad=false"],
}
HEADERS = ["internal.h", "ptx.cuh", "gemm_skinny.cuh", "gemm_w4a16.cuh", "mx_block.cuh"]


def _mtime(path: str) -> float:
    return os.path.getmtime(path) if os.path.exists(path) else 0.0


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    deps = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "macaq.h")]
    newest_dep = max(_mtime(d) for d in deps)
    objs = []
    for unit, extra in UNITS.items():
        src = os.path.join(CSRC, unit)
        obj = os.path.join(BUILD, unit.replace(".cu", ".o"))
        objs.append(obj)
        if force or _mtime(obj) < max(_mtime(src), newest_dep):
            cmd = [NVCC, *COMMON, *ARCH, *extra, "-c", src, "-o", obj]
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            subprocess.check_call(cmd)
    if force or _mtime(LIB) < max(_mtime(o) for o in objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [NVCC, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-cudart", "static", "-o", tmp, *objs]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        subprocess.check_call(cmd)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
