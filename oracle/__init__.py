"""Oracle for the ZeRO sharded optimizer step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never imports, links or calls it.

``zero_oracle.c`` is a plain single-threaded C restatement of the step (see
its header for the passages it follows); this module compiles it with gcc
(``-O2 -ffp-contract=off``, no fast-math) and exposes it through ctypes on
numpy arrays.  ``memory`` holds the closed forms of the memory and
communication accounting.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from . import memory  # noqa: F401  (re-exported)

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "zero_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

F32, BF16, F16 = 0, 1, 2
NP_STORAGE = {F32: np.float32, BF16: np.uint16, F16: np.uint16}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to its source when missing or stale."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
           "-Wall", "-fPIC", "-shared", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


def load(path: str) -> ctypes.CDLL:
    """Open an oracle library at `path` with its function signatures."""
    L = ctypes.CDLL(path)
    i64, i32, f32, f64 = ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_double
    vp, fp = ctypes.c_void_p, ctypes.POINTER(ctypes.c_float)
    vpp = ctypes.POINTER(ctypes.c_void_p)
    i64p = ctypes.POINTER(ctypes.c_int64)
    sig = {
        "orc_shard_size": (i64, [i64, i32]),
        "orc_owner": (i32, [i64, i64, i32]),
        "orc_elem_size": (i32, [i32]),
        "orc_widen_array": (None, [vp, i32, i64, fp]),
        "orc_cast": (None, [fp, i64, i32, vp]),
        "orc_rank_sum": (None, [vpp, i32, i32, i64, i64, fp]),
        "orc_reduce_scatter_sum": (ctypes.c_int, [vpp, i32, i64, i32, i32, fp, i64p]),
        "orc_average": (i64, [fp, i64, i32, f32, fp]),
        "orc_all_gather": (None, [vpp, i32, i64, i32, vp, i64p]),
        "orc_all_reduce_mean": (None, [vpp, i32, i64, i32, fp]),
        "orc_adam_scalars": (None, [f64, f64, i64, fp]),
        "orc_adam": (None, [fp, fp, fp, fp, i64, f64, f64, f64, f64, i64, f64]),
        "orc_zero_step": (ctypes.c_int, [vpp, i32, i64, i32, fp, fp, fp, vp, i32,
                                         f64, f64, f64, f64, i64, f32, fp, i64p, f64]),
        "orc_zero_rank_step": (ctypes.c_int, [vpp, i32, i64, i32, i32, fp, fp, fp,
                                              vp, i32, f64, f64, f64, f64, i64, f32,
                                              i64, fp, i64p, f64]),
        "orc_scale_update": (f32, [f32, i32, i64p, i64]),
        "orc_row_shard_size": (i64, [i64, i64, i32]),
        "orc_zero_step_s": (ctypes.c_int, [vpp, i32, i64, i32, i64, fp, fp, fp, vp, i32,
                                           f64, f64, f64, f64, i64, f32, fp, i64p, f64]),
        "orc_zero_rank_step_s": (ctypes.c_int, [vpp, i32, i64, i32, i64, i32, fp, fp, fp,
                                                vp, i32, f64, f64, f64, f64, i64, f32,
                                                i64, fp, i64p, f64]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            # a copy of the oracle with a planted mistake, for the tests that
            # check the pins catch it
            override = os.environ.get("ZERO_ORACLE_LIB")
            if override:
                _lib = load(override)
            else:
                build()
                _lib = load(LIB)
    return _lib


def use_library(L) -> ctypes.CDLL:
    """Swap the library every oracle function calls (None: back to the
    built one); returns the previous one.  For the tests that plant
    mistakes in copies of the oracle."""
    global _lib
    with _lock:
        prev, _lib = _lib, L
    return prev


# ----------------------------------------------------------------- helpers

def _fp(a: np.ndarray):
    assert a.dtype == np.float32 and a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def _vp(a: np.ndarray):
    assert a.flags.c_contiguous
    return ctypes.c_void_p(a.ctypes.data)


def _ptrs(arrs):
    for a in arrs:
        assert a.flags.c_contiguous
    return (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])


def _check(arr: np.ndarray, dtype: int):
    if arr.dtype != NP_STORAGE[dtype]:
        raise TypeError("expected %s storage for dtype code %d, got %s"
                        % (NP_STORAGE[dtype], dtype, arr.dtype))


def shard_size(numel: int, world: int) -> int:
    return int(lib().orc_shard_size(numel, world))


def owner(i: int, numel: int, world: int) -> int:
    return int(lib().orc_owner(i, numel, world))


def widen(arr: np.ndarray, dtype: int) -> np.ndarray:
    _check(arr, dtype)
    out = np.empty(arr.size, np.float32)
    lib().orc_widen_array(_vp(arr), dtype, arr.size, _fp(out))
    return out


def cast(x: np.ndarray, dtype: int) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float32)
    out = np.empty(x.size, NP_STORAGE[dtype])
    lib().orc_cast(_fp(x), x.size, dtype, _vp(out))
    return out


def rank_sum(bufs, dtype: int, n: int, n_valid: int) -> np.ndarray:
    for b in bufs:
        _check(b, dtype)
        assert b.size >= min(n, n_valid)
    acc = np.empty(n, np.float32)
    lib().orc_rank_sum(_ptrs(bufs), dtype, len(bufs), n, n_valid, _fp(acc))
    return acc


def reduce_scatter_sum(grads, dtype: int, numel: int, rank: int, bytes_sent=None):
    world = len(grads)
    for g in grads:
        _check(g, dtype)
        assert g.size >= numel
    S = shard_size(numel, world)
    out = np.empty(S, np.float32)
    bs = np.zeros(world, np.int64) if bytes_sent is None else bytes_sent
    rc = lib().orc_reduce_scatter_sum(_ptrs(grads), dtype, numel, world, rank, _fp(out),
                                      bs.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)))
    assert rc == 0
    return out


def average(acc: np.ndarray, world: int, loss_scale: float = 0.0):
    acc = np.ascontiguousarray(acc, np.float32)
    g = np.empty_like(acc)
    bad = lib().orc_average(_fp(acc), acc.size, world, loss_scale, _fp(g))
    return g, int(bad)


def all_gather(shards, dtype: int, bytes_sent=None) -> np.ndarray:
    world = len(shards)
    S = shards[0].size
    for s in shards:
        _check(s, dtype)
        assert s.size == S
    full = np.empty(world * S, NP_STORAGE[dtype])
    bs = np.zeros(world, np.int64) if bytes_sent is None else bytes_sent
    lib().orc_all_gather(_ptrs(shards), dtype, S, world, _vp(full),
                         bs.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)))
    return full


def all_reduce_mean(grads, dtype: int, numel: int) -> np.ndarray:
    world = len(grads)
    for g in grads:
        _check(g, dtype)
    P = shard_size(numel, world) * world
    out = np.empty(P, np.float32)
    lib().orc_all_reduce_mean(_ptrs(grads), dtype, numel, world, _fp(out))
    return out


def adam_scalars(beta1: float, beta2: float, t: int):
    out = np.empty(4, np.float32)
    lib().orc_adam_scalars(beta1, beta2, t, _fp(out))
    return out


def adam(x, m, v, g, lr, beta1, beta2, eps, t, weight_decay=0.0):
    """In-place Adam (AdamW when weight_decay != 0) on float32 arrays x, m, v
    with gradient g."""
    for a in (x, m, v, g):
        assert a.dtype == np.float32 and a.size == x.size
    lib().orc_adam(_fp(x), _fp(m), _fp(v), _fp(np.ascontiguousarray(g)), x.size,
                   lr, beta1, beta2, eps, t, weight_decay)


def row_shard_size(rows: int, row_elems: int, world: int) -> int:
    """Shard length of FSDP2's dim-0 layout: ceil(rows/world) whole rows."""
    return int(lib().orc_row_shard_size(rows, row_elems, world))


def zero_step(grads, grad_dtype, numel, master, m, v, full, param_dtype,
              lr, beta1, beta2, eps, t, loss_scale=0.0, weight_decay=0.0, shard=None):
    """All-ranks ZeRO-2 step, in place.  Returns (skipped, n_nonfinite).
    `shard` overrides the shard length ceil(numel/N) (the dim-0 layout)."""
    world = len(grads)
    for g in grads:
        _check(g, grad_dtype)
        assert g.size >= numel
    S = shard_size(numel, world) if shard is None else shard
    P = S * world
    for a in (master, m, v):
        assert a.dtype == np.float32 and a.size == P
    _check(full, param_dtype)
    assert full.size == P
    work = np.empty(2 * P + 16, np.float32)
    bad = ctypes.c_int64(0)
    rc = lib().orc_zero_step_s(_ptrs(grads), grad_dtype, numel, world, S, _fp(master), _fp(m),
                               _fp(v), _vp(full), param_dtype, lr, beta1, beta2, eps, t,
                               loss_scale, _fp(work), ctypes.byref(bad), weight_decay)
    if rc < 0:
        raise ValueError("orc_zero_step: bad arguments")
    return bool(rc == 1), int(bad.value)


def zero_rank_step(slices, grad_dtype, numel, rank, master, m, v, lp_out, param_dtype,
                   lr, beta1, beta2, eps, t, loss_scale=0.0, others_nonfinite=0,
                   weight_decay=0.0, shard=None):
    """One rank's view, in place.  Returns (skipped, n_nonfinite_local).
    `shard` overrides the shard length ceil(numel/N) (the dim-0 layout)."""
    world = len(slices)
    S = shard_size(numel, world) if shard is None else shard
    for s in slices:
        _check(s, grad_dtype)
        assert s.size == S
    for a in (master, m, v):
        assert a.dtype == np.float32 and a.size == S
    _check(lp_out, param_dtype)
    assert lp_out.size == S and lp_out.flags.c_contiguous
    work = np.empty(max(S, 1), np.float32)
    bad = ctypes.c_int64(0)
    rc = lib().orc_zero_rank_step_s(_ptrs(slices), grad_dtype, numel, world, S, rank,
                                    _fp(master), _fp(m), _fp(v), _vp(lp_out), param_dtype, lr,
                                    beta1, beta2, eps, t, loss_scale, others_nonfinite, _fp(work),
                                    ctypes.byref(bad), weight_decay)
    if rc < 0:
        raise ValueError("orc_zero_rank_step: bad arguments")
    return bool(rc == 1), int(bad.value)


def scale_update(scale: float, skipped: bool, good_steps: int, growth_interval: int):
    gs = ctypes.c_int64(good_steps)
    new = lib().orc_scale_update(scale, int(skipped), ctypes.byref(gs), growth_interval)
    return float(new), int(gs.value)
