"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

Holds none of the method's arithmetic: only the counter-based generator of
gradients and initial weights defined in ``synth.cu`` (splitmix64 words summed
Irwin-Hall style into an approximately normal integer, times one fp32 scale,
rounded to the buffer's type).  ``np_fill`` restates the same definition in
numpy so the C version can be checked on a CPU.

Streams are named by a tag: (kind, step, rank, unit).  ``KIND_MASTER`` draws
initial fp32 master weights, ``KIND_GRAD`` rank `rank`'s local gradient at
iteration `step`; index i is the element's flat position (within its unit).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "synth.cu")
LIB = os.path.join(HERE, "libsynth.so")

KIND_MASTER, KIND_GRAD, KIND_PICK = 0, 1, 2
F32, BF16, F16 = 0, 1, 2
NP_STORAGE = {F32: np.float32, BF16: np.uint16, F16: np.uint16}
IH_STD = math.sqrt((65536.0 ** 2 - 1.0) / 3.0)

_lock = threading.Lock()
_lib = None


def build_cmd(out: str):
    return ["nvcc", "-O2", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
            "-gencode", "arch=compute_103a,code=sm_103a", "-cudart", "static",
            "-o", out, SRC]


def build(force: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    subprocess.run(build_cmd(tmp), check=True)
    os.replace(tmp, LIB)
    return LIB


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(LIB)
            u64, i64, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
            L.synth_tag.restype = u64
            L.synth_tag.argtypes = [i64, i64, i64, i64]
            L.synth_key.restype = u64
            L.synth_key.argtypes = [u64, u64]
            L.synth_word.restype = u64
            L.synth_word.argtypes = [u64, i64]
            L.synth_pick_index.restype = i64
            L.synth_pick_index.argtypes = [u64, i64]
            L.synth_fill_host.restype = None
            L.synth_fill_host.argtypes = [vp, ctypes.c_int, i64, i64, vp, u64, ctypes.c_float]
            L.synth_fill_device.restype = ctypes.c_int
            L.synth_fill_device.argtypes = [vp, ctypes.c_int, i64, i64, vp, u64,
                                            ctypes.c_float, vp]
            _lib = L
    return _lib


def scale_for(sigma: float) -> float:
    """fp32 scale turning the centred Irwin-Hall integer into N(0, sigma^2)."""
    return float(np.float32(sigma / IH_STD))


def key(seed: int, kind: int, step: int = 0, rank: int = 0, unit: int = 0) -> int:
    L = lib()
    return int(L.synth_key(seed, L.synth_tag(kind, step, rank, unit)))


def pick_index(seed: int, n: int, step: int = 0, rank: int = 0, unit: int = 0) -> int:
    return int(lib().synth_pick_index(key(seed, KIND_PICK, step, rank, unit), n))


def fill_host(n: int, dtype: int, k: int, sigma: float, index0: int = 0,
              indices: np.ndarray | None = None) -> np.ndarray:
    """n draws of stream `k` (a key) on the host, in the storage of `dtype`."""
    out = np.empty(n, NP_STORAGE[dtype])
    idx = None
    if indices is not None:
        indices = np.ascontiguousarray(indices, np.int64)
        assert indices.size == n
        idx = ctypes.c_void_p(indices.ctypes.data)
    lib().synth_fill_host(ctypes.c_void_p(out.ctypes.data), dtype, n, index0, idx, k,
                          scale_for(sigma))
    return out


def fill_device(ptr: int, n: int, dtype: int, k: int, sigma: float, stream: int,
                index0: int = 0, indices_ptr: int | None = None) -> None:
    """The same draws written to device memory at `ptr`, on `stream`."""
    rc = lib().synth_fill_device(ctypes.c_void_p(ptr), dtype, n, index0,
                                 ctypes.c_void_p(indices_ptr) if indices_ptr else None,
                                 k, scale_for(sigma), ctypes.c_void_p(stream))
    if rc != 0:
        raise RuntimeError("synth_fill_device failed: cudaError %d" % rc)


# ----------------------------------------------- numpy restatement (checks)

_M64 = (1 << 64) - 1


def _np_mix64(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * np.uint64(0xBF58476D1CE4E5B9)
    z = z ^ (z >> np.uint64(27))
    z = z * np.uint64(0x94D049BB133111EB)
    z = z ^ (z >> np.uint64(31))
    return z


def _py_mix64(z: int) -> int:
    z &= _M64
    z ^= z >> 30
    z = (z * 0xBF58476D1CE4E5B9) & _M64
    z ^= z >> 27
    z = (z * 0x94D049BB133111EB) & _M64
    z ^= z >> 31
    return z


def py_key(seed: int, kind: int, step: int = 0, rank: int = 0, unit: int = 0) -> int:
    tag = (step << 36) | ((rank & 0xFFFF) << 20) | ((unit & 0xFFFF) << 4) | (kind & 0xF)
    return _py_mix64(_py_mix64(tag) ^ seed)


def _np_bf16_bits(x: np.ndarray) -> np.ndarray:
    u = x.astype(np.float32).view(np.uint32).astype(np.uint64)
    hi = u >> np.uint64(16)
    lo = u & np.uint64(0xFFFF)
    up = (lo > 0x8000) | ((lo == 0x8000) & ((hi & np.uint64(1)) == 1))
    hi = hi + up.astype(np.uint64)
    nan = (u & np.uint64(0x7FFFFFFF)) > np.uint64(0x7F800000)
    hi = np.where(nan, (u >> np.uint64(16)) | np.uint64(0x40), hi)
    return hi.astype(np.uint16)


def np_fill(n: int, dtype: int, k: int, sigma: float, index0: int = 0,
            indices: np.ndarray | None = None) -> np.ndarray:
    """Pure-numpy restatement of ``fill_host`` (slow; for checks)."""
    if indices is None:
        i = np.arange(index0, index0 + n, dtype=np.int64)
    else:
        i = np.asarray(indices, np.int64)
    with np.errstate(over="ignore"):
        w = _np_mix64(np.uint64(k) + (i + 1).astype(np.uint64) * np.uint64(0x9E3779B97F4A7C15))
    s = np.zeros(n, np.int64)
    for q in range(4):
        s += ((w >> np.uint64(16 * q)) & np.uint64(0xFFFF)).astype(np.int64)
    c = (s - 131070).astype(np.float32)
    x = (c * np.float32(scale_for(sigma))).astype(np.float32)
    if dtype == F32:
        return x
    if dtype == F16:
        return x.astype(np.float16).view(np.uint16)
    return _np_bf16_bits(x)
