"""ctypes wrapper of the compute stand-in used by the ZeRO-3 overlap
measurement (libstandin.so, built next to its source)."""
from __future__ import annotations

import ctypes
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "standin.cu")
LIB = os.path.join(HERE, "libstandin.so")
_lib = None


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    subprocess.run(["nvcc", "-O3", "-Xcompiler", "-fPIC", "-shared", "-gencode",
                    "arch=compute_103a,code=sm_103a", "-cudart", "static", "-o", tmp, SRC],
                   check=True)
    os.replace(tmp, LIB)
    return LIB


def busy(sink_ptr: int, blocks: int, iters: int, stream: int) -> None:
    global _lib
    if _lib is None:
        build()
        _lib = ctypes.CDLL(LIB)
        _lib.standin_busy.restype = ctypes.c_int
        _lib.standin_busy.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                      ctypes.c_void_p]
    rc = _lib.standin_busy(ctypes.c_void_p(sink_ptr), blocks, iters, ctypes.c_void_p(stream))
    if rc != 0:
        raise RuntimeError("standin_busy failed: cudaError %d" % rc)
