"""Build libzero.so, the CUDA library behind the binding, for sm_103a.

Each translation unit is compiled in parallel with nvcc, then linked into a
shared library next to this file (in-tree, so the binding finds it).  No
fast-math and no flush-to-zero: the step's numerics are defined operation by
operation, and -fmad=false keeps any multiply-add from being fused.
"""
from __future__ import annotations

import concurrent.futures
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libzero.so")
SOURCES = ["zero_abi.cu", "zero_step_kernels.cu", "zero_gather.cu", "zero_advance.cu"]
HEADERS = ["zero_internal.h", "zero_row_copy.cuh", os.path.join("..", "..", "include", "zero.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-fmad=false", "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
              "-Xcompiler", "-Wall"] + ARCH


def _newest_input() -> float:
    paths = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.abspath(__file__)]
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _newest_input():
        return LIB
    os.makedirs(BUILD, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        cmd = ["nvcc", *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        subprocess.run(cmd, check=True)
        return obj

    with concurrent.futures.ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + ".tmp.%d" % os.getpid()
    subprocess.run(["nvcc", "-shared", *ARCH, "-cudart", "static", "-o", tmp, *objs], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
    print(LIB)
