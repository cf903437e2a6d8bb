"""Thin ctypes binding of libzero.so: the same entry points under the same
names, with Python-side argument marshalling only (torch tensors or ints for
device pointers, torch streams or ints for CUDA streams, lists for pointer
arrays).  Every step of the computation runs in the library's CUDA kernels;
there is no fallback: if the library is missing, importing this module
raises.  Negative return codes raise ZeroError with the library's message.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libzero.so")

ZERO_F32, ZERO_BF16, ZERO_F16 = 0, 1, 2
ZERO_OK, ZERO_SKIPPED = 0, 1
ZERO_EINVAL, ZERO_ECUDA, ZERO_EALIGN, ZERO_ESTATE, ZERO_ETIMEOUT = -1, -2, -3, -4, -5
ZERO_MAX_RANKS = 256
ZERO_HYPER_BYTES = 128
ZERO_GATHER_FAST, ZERO_GATHER_LEAN = 0, 1


class ZeroError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__("%s (%d): %s" % (_strerror(code), code, message))
        self.code = code


if not os.path.exists(LIB_PATH):
    raise ImportError("libzero.so is not built (run __graft_entry__.build() or "
                      "python zero_sharded_optimizer_step_gb300/build.py): %s" % LIB_PATH)

_L = ctypes.CDLL(LIB_PATH)

_i32, _i64, _u64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64
_f32, _f64, _vp = ctypes.c_float, ctypes.c_double, ctypes.c_void_p
_vpp = ctypes.POINTER(ctypes.c_void_p)
_ctxp = ctypes.c_void_p

_SIGS = {
    "zero_shard_size": (_i64, [_i64, _i32]),
    "zero_model_state_bytes": (_f64, [_i64, _i32, _i32]),
    "zero_scale_update": (_f32, [_f32, _i32, ctypes.POINTER(_i64), _i64]),
    "zero_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "zero_last_error": (ctypes.c_char_p, []),
    "zero_init": (ctypes.c_int, [ctypes.POINTER(_ctxp), _i64, _i32, _i32, _i32, _i32, _i32,
                                 ctypes.POINTER(_i64), _i32]),
    "zero_init_ranks": (ctypes.c_int, [ctypes.POINTER(_ctxp), _i64, _i32, _i32, _i32, _i32,
                                       _i32, _i32, ctypes.POINTER(_i64), _i32]),
    "zero_init_dim0": (ctypes.c_int, [ctypes.POINTER(_ctxp), _i32, _i32, _i32, _i32,
                                      ctypes.POINTER(_i64), ctypes.POINTER(_i64), _i32]),
    "zero_destroy": (ctypes.c_int, [_ctxp]),
    "zero_ctx_shard_size": (_i64, [_ctxp, _i32]),
    "zero_ctx_state_elems": (_i64, [_ctxp]),
    "zero_ctx_param_elems": (_i64, [_ctxp]),
    "zero_ctx_unit_state_offset": (_i64, [_ctxp, _i32]),
    "zero_ctx_unit_param_offset": (_i64, [_ctxp, _i32]),
    "zero_state_bytes": (_i64, [_ctxp]),
    "zero_bind": (ctypes.c_int, [_ctxp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "zero_bind_allreduce_out": (ctypes.c_int, [_ctxp, _vp]),
    "zero_set_weight_decay": (ctypes.c_int, [_ctxp, _f64]),
    "zero_bind_hyper": (ctypes.c_int, [_ctxp, _vp]),
    "zero_hyper_slot": (ctypes.c_int, [_ctxp, ctypes.POINTER(_vp)]),
    "zero_load_hyper": (ctypes.c_int, [_ctxp, _vp, _vp]),
    "zero_prepare_step": (ctypes.c_int, [_ctxp, _vp, _f64, _f64, _f64, _f64, _i64, _f32]),
    "zero_set_gather_mode": (ctypes.c_int, [_ctxp, _i32]),
    "zero_advance_table_bytes": (_i64, [_i64]),
    "zero_fill_advance_table": (ctypes.c_int, [_vp, _i64, _f64, _f64]),
    "zero_advance_state": (ctypes.c_int, [_vp, _i64, _f32, _i64]),
    "zero_bind_advance": (ctypes.c_int, [_ctxp, _vp, _i64, _vp]),
    "zero_advance_step": (ctypes.c_int, [_ctxp, _vp]),
    "zero_gather_timeouts": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32)]),
    "zero_set_gather_wait_polls": (ctypes.c_int, [ctypes.c_int64]),
    "zero_set_step_occupancy": (ctypes.c_int, [_ctxp, _i32]),
    "zero_bind_shadow": (ctypes.c_int, [_ctxp, _vp, _vp, _vp, _vp]),
    "zero_current_state": (ctypes.c_int, [_ctxp, ctypes.POINTER(_i32)]),
    "zero_step": (ctypes.c_int, [_ctxp, _vpp, _i32, _f64, _f64, _f64, _f64, _i64, _f32, _vp]),
    "zero_step_reduce": (ctypes.c_int, [_ctxp, _vpp, _i32, _f32, _vp]),
    "zero_step_apply": (ctypes.c_int, [_ctxp, _f64, _f64, _f64, _f64, _i64, _vp]),
    "zero_bucket_begin": (ctypes.c_int, [_ctxp, _f32]),
    "zero_bucket_step": (ctypes.c_int, [_ctxp, _i64, _i64, _vpp, _i32, _f64, _f64, _f64, _f64,
                                        _i64, _vp]),
    "zero_bucket_end": (ctypes.c_int, [_ctxp, _f64, _f64, _f64, _f64, _i64, _vp]),
    "zero_step_status": (ctypes.c_int, [_ctxp, ctypes.POINTER(_i32), ctypes.POINTER(_i32)]),
    "zero_step_id": (_u64, [_ctxp]),
    "zero_allgather": (ctypes.c_int, [_ctxp, _vpp, _i32, _vp, _i32, _vp]),
    "zero3_begin_step": (ctypes.c_int, [_ctxp]),
    "zero3_begin_step_scaled": (ctypes.c_int, [_ctxp, _f32]),
    "zero3_end_step": (ctypes.c_int, [_ctxp, _vp]),
    "zero3_gather_unit": (ctypes.c_int, [_ctxp, _i32, _vpp, _i32, _vp, _vp]),
    "zero3_step_unit": (ctypes.c_int, [_ctxp, _i32, _vpp, _i32, _f64, _f64, _f64, _f64, _i64,
                                       _vp]),
    "zero3_reduce_unit": (ctypes.c_int, [_ctxp, _i32, _vpp, _i32, _f32, _vp]),
    "zero3_step_unit_gather": (ctypes.c_int, [_ctxp, _i32, _vpp, _i32, _f64, _f64, _f64, _f64,
                                              _i64, _i32, _vpp, _i32, _vp, _vp]),
    "zero3_step_units_gather": (ctypes.c_int, [_ctxp, _i32, _i32, _vpp, _i32, _f64, _f64, _f64,
                                               _f64, _i64, _i32, _i32, _vpp, _i32, _vpp, _vp]),
    "zero3_gather_group": (ctypes.c_int, [_ctxp, _i32, _i32, _vpp, _i32, _vpp, _vp]),
    "zero3_step_group": (ctypes.c_int, [_ctxp, _i32, _i32, _vpp, _i32, _f64, _f64, _f64, _f64,
                                        _i64, _vp]),
    "zero3_reduce_group": (ctypes.c_int, [_ctxp, _i32, _i32, _vpp, _i32, _f32, _vp]),
    "zero_step_noalloc": (ctypes.c_int, [_ctxp, _vpp, _i32, _f64, _f64, _f64, _f64, _i64, _f32,
                                         _vp]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_L, _name)
    _fn.restype = _res
    _fn.argtypes = _args

EXPORTED = tuple(_SIGS)


def _strerror(code: int) -> str:
    return _L.zero_strerror(code).decode()


def _check(rc: int) -> int:
    if rc < 0:
        raise ZeroError(rc, _L.zero_last_error().decode())
    return rc


def _ptr(x) -> int | None:
    """Device address of a tensor, an int address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _ptrs(xs):
    if xs is None:
        return None
    return (ctypes.c_void_p * len(xs))(*[_ptr(x) for x in xs])


def _stream(s) -> int | None:
    if s is None:
        try:
            import torch
            return torch.cuda.current_stream().cuda_stream
        except Exception:
            return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


class Ctx:
    """Owner of one zero_ctx handle (zero_destroy on close / collection)."""

    def __init__(self, handle: int):
        self.handle = handle

    def close(self):
        if self.handle:
            _L.zero_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _h(ctx) -> int:
    h = ctx.handle if isinstance(ctx, Ctx) else ctx
    if not h:
        raise ZeroError(ZERO_EINVAL, "closed or null context")
    return h


# ------------------------------------------------------------ host only

def zero_shard_size(numel: int, world: int) -> int:
    return _L.zero_shard_size(numel, world)


def zero_model_state_bytes(numel: int, world: int, stage: int) -> float:
    return _L.zero_model_state_bytes(numel, world, stage)


def zero_scale_update(scale: float, skipped: bool, good_steps: int, growth_interval: int):
    """Returns (new_scale, new_good_steps)."""
    gs = _i64(good_steps)
    s = _L.zero_scale_update(scale, int(bool(skipped)), ctypes.byref(gs), growth_interval)
    return float(s), int(gs.value)


def zero_strerror(code: int) -> str:
    return _strerror(code)


def zero_last_error() -> str:
    return _L.zero_last_error().decode()


# -------------------------------------------------------------- context

def zero_init(numel: int, world: int, stage: int, grad_dtype: int, param_dtype: int,
              rank: int = -1, unit_numels=None) -> Ctx:
    h = _ctxp()
    units = None
    n_units = 0
    if unit_numels is not None:
        n_units = len(unit_numels)
        units = (_i64 * n_units)(*unit_numels)
    _check(_L.zero_init(ctypes.byref(h), numel, world, stage, grad_dtype, param_dtype, rank,
                        units, n_units))
    return Ctx(h.value)


def zero_init_ranks(numel: int, world: int, stage: int, grad_dtype: int, param_dtype: int,
                    first_rank: int, n_ranks: int, unit_numels=None) -> Ctx:
    """A view of ranks [first_rank, first_rank + n_ranks) (stage 3: of each
    unit)."""
    h = _ctxp()
    units = None
    n_units = 0
    if unit_numels is not None:
        n_units = len(unit_numels)
        units = (_i64 * n_units)(*unit_numels)
    _check(_L.zero_init_ranks(ctypes.byref(h), numel, world, stage, grad_dtype, param_dtype,
                              first_rank, n_ranks, units, n_units))
    return Ctx(h.value)


def zero_init_dim0(world: int, grad_dtype: int, param_dtype: int, rank: int, shapes) -> Ctx:
    """Stage 3 in FSDP2's dim-0 layout; shapes = [(rows, row_elems), ...]."""
    h = _ctxp()
    n = len(shapes)
    rows = (_i64 * n)(*[r for r, _ in shapes])
    elems = (_i64 * n)(*[e for _, e in shapes])
    _check(_L.zero_init_dim0(ctypes.byref(h), world, grad_dtype, param_dtype, rank, rows,
                             elems, n))
    return Ctx(h.value)


def zero_destroy(ctx: Ctx) -> None:
    ctx.close()


def zero_ctx_shard_size(ctx, unit: int = -1) -> int:
    return _L.zero_ctx_shard_size(_h(ctx), unit)


def zero_ctx_state_elems(ctx) -> int:
    return _L.zero_ctx_state_elems(_h(ctx))


def zero_ctx_param_elems(ctx) -> int:
    return _L.zero_ctx_param_elems(_h(ctx))


def zero_ctx_unit_state_offset(ctx, unit: int) -> int:
    return _L.zero_ctx_unit_state_offset(_h(ctx), unit)


def zero_ctx_unit_param_offset(ctx, unit: int) -> int:
    return _L.zero_ctx_unit_param_offset(_h(ctx), unit)


def zero_state_bytes(ctx) -> int:
    return _L.zero_state_bytes(_h(ctx))


def zero_bind(ctx, master, m, v, params, g_scratch=None, flag=None) -> None:
    _check(_L.zero_bind(_h(ctx), _ptr(master), _ptr(m), _ptr(v), _ptr(params),
                        _ptr(g_scratch), _ptr(flag)))


def zero_bind_shadow(ctx, master_b, m_b, v_b, cur) -> None:
    _check(_L.zero_bind_shadow(_h(ctx), _ptr(master_b), _ptr(m_b), _ptr(v_b), _ptr(cur)))


def zero_current_state(ctx) -> int:
    """Synchronizes; 0 = the zero_bind state set is current, 1 = the second."""
    w = _i32(0)
    _check(_L.zero_current_state(_h(ctx), ctypes.byref(w)))
    return int(w.value)


def zero_set_gather_mode(ctx, mode: int) -> None:
    _check(_L.zero_set_gather_mode(_h(ctx), mode))


def zero_gather_timeouts() -> int:
    """The count of lean-gather waits that ran out (ZERO_ETIMEOUT from the C
    call when it is not 0; the count is returned either way)."""
    c = ctypes.c_uint32(0)
    rc = _L.zero_gather_timeouts(ctypes.byref(c))
    if rc != ZERO_ETIMEOUT:
        _check(rc)
    return int(c.value)


def zero_set_step_occupancy(ctx, blocks_per_sm: int) -> None:
    """At most blocks_per_sm step-kernel blocks per SM (0: as many as fit)."""
    _check(_L.zero_set_step_occupancy(_h(ctx), blocks_per_sm))


def zero_set_gather_wait_polls(polls: int) -> None:
    """Polls of the lean gather's first wait on each tile; 0 makes the waits
    run out (a test of the timeout path), < 0 restores the default."""
    _check(_L.zero_set_gather_wait_polls(polls))


def zero_bind_hyper(ctx, d_hyper) -> None:
    _check(_L.zero_bind_hyper(_h(ctx), _ptr(d_hyper)))


def zero_load_hyper(ctx, host_block, stream=None) -> None:
    _check(_L.zero_load_hyper(_h(ctx), _ptr(host_block), _stream(stream)))


def zero_hyper_slot(ctx) -> int:
    """Device address (int) of the context's constant slot for its scalar block."""
    p = _vp()
    _check(_L.zero_hyper_slot(_h(ctx), ctypes.byref(p)))
    return int(p.value)


def zero_prepare_step(ctx, host_hyper, lr: float, beta1: float, beta2: float, eps: float,
                      t: int, loss_scale: float = 0.0) -> None:
    """host_hyper: a host buffer of ZERO_HYPER_BYTES (a pinned uint8 tensor or an
    int address)."""
    _check(_L.zero_prepare_step(_h(ctx), _ptr(host_hyper), lr, beta1, beta2, eps, t,
                                loss_scale))


ZERO_ADVANCE_STATE_BYTES = 32


def zero_advance_table_bytes(t_max: int) -> int:
    return int(_L.zero_advance_table_bytes(t_max))


def zero_fill_advance_table(host_table, t_max: int, beta1: float, beta2: float) -> None:
    """host_table: a host buffer of zero_advance_table_bytes(t_max) bytes."""
    _check(_L.zero_fill_advance_table(_ptr(host_table), t_max, beta1, beta2))


def zero_advance_state(host_state, t: int, loss_scale: float, growth_interval: int) -> None:
    """host_state: a host buffer of ZERO_ADVANCE_STATE_BYTES bytes."""
    _check(_L.zero_advance_state(_ptr(host_state), t, loss_scale, growth_interval))


def zero_bind_advance(ctx, d_table, t_max: int, d_state) -> None:
    _check(_L.zero_bind_advance(_h(ctx), _ptr(d_table), t_max, _ptr(d_state)))


def zero_advance_step(ctx, stream=None) -> None:
    _check(_L.zero_advance_step(_h(ctx), _stream(stream)))


def zero_set_weight_decay(ctx, weight_decay: float) -> None:
    _check(_L.zero_set_weight_decay(_h(ctx), weight_decay))


def zero_bind_allreduce_out(ctx, grad_avg) -> None:
    _check(_L.zero_bind_allreduce_out(_h(ctx), _ptr(grad_avg)))


# ------------------------------------------------------------- the step

def zero_step(ctx, grads, lr: float, beta1: float, beta2: float, eps: float, t: int,
              loss_scale: float = 0.0, stream=None) -> None:
    _check(_L.zero_step(_h(ctx), _ptrs(grads), len(grads), lr, beta1, beta2, eps, t,
                        loss_scale, _stream(stream)))


def zero_step_reduce(ctx, grads, loss_scale: float = 0.0, stream=None) -> None:
    _check(_L.zero_step_reduce(_h(ctx), _ptrs(grads), len(grads), loss_scale, _stream(stream)))


def zero_step_apply(ctx, lr: float, beta1: float, beta2: float, eps: float, t: int,
                    stream=None) -> None:
    _check(_L.zero_step_apply(_h(ctx), lr, beta1, beta2, eps, t, _stream(stream)))


def zero_bucket_begin(ctx, loss_scale: float = 0.0) -> None:
    _check(_L.zero_bucket_begin(_h(ctx), loss_scale))


def zero_bucket_step(ctx, offset: int, count: int, grads, lr: float, beta1: float, beta2: float,
                     eps: float, t: int, stream=None) -> None:
    _check(_L.zero_bucket_step(_h(ctx), offset, count, _ptrs(grads), len(grads), lr, beta1,
                               beta2, eps, t, _stream(stream)))


def zero_bucket_end(ctx, lr: float, beta1: float, beta2: float, eps: float, t: int,
                    stream=None) -> None:
    _check(_L.zero_bucket_end(_h(ctx), lr, beta1, beta2, eps, t, _stream(stream)))


def zero_step_status(ctx):
    """Synchronizes; returns (nonfinite, skipped) as bools."""
    nf, sk = _i32(0), _i32(0)
    _check(_L.zero_step_status(_h(ctx), ctypes.byref(nf), ctypes.byref(sk)))
    return bool(nf.value), bool(sk.value)


def zero_step_id(ctx) -> int:
    return int(_L.zero_step_id(_h(ctx)))


def zero_allgather(ctx, shards, full, dtype: int, stream=None) -> None:
    _check(_L.zero_allgather(_h(ctx), _ptrs(shards), len(shards), _ptr(full), dtype,
                             _stream(stream)))


# -------------------------------------------------------------- stage 3

def zero3_begin_step(ctx) -> None:
    _check(_L.zero3_begin_step(_h(ctx)))


def zero3_begin_step_scaled(ctx, loss_scale: float) -> None:
    _check(_L.zero3_begin_step_scaled(_h(ctx), loss_scale))


def zero3_end_step(ctx, stream=None) -> None:
    _check(_L.zero3_end_step(_h(ctx), _stream(stream)))


def zero3_gather_unit(ctx, unit: int, shards, unit_full, stream=None) -> None:
    _check(_L.zero3_gather_unit(_h(ctx), unit, _ptrs(shards), len(shards), _ptr(unit_full),
                                _stream(stream)))


def zero3_step_unit(ctx, unit: int, grads, lr: float, beta1: float, beta2: float, eps: float,
                    t: int, stream=None) -> None:
    _check(_L.zero3_step_unit(_h(ctx), unit, _ptrs(grads), len(grads), lr, beta1, beta2, eps,
                              t, _stream(stream)))


def zero3_step_unit_gather(ctx, unit: int, grads, lr: float, beta1: float, beta2: float,
                           eps: float, t: int, gather_unit: int, shards, unit_full,
                           stream=None) -> None:
    """One backward visit: unit `unit`'s step and unit `gather_unit`'s gather."""
    _check(_L.zero3_step_unit_gather(_h(ctx), unit, _ptrs(grads), len(grads), lr, beta1, beta2,
                                     eps, t, gather_unit, _ptrs(shards), len(shards),
                                     _ptr(unit_full), _stream(stream)))


def zero3_step_units_gather(ctx, first_unit: int, grads, lr: float, beta1: float, beta2: float,
                            eps: float, t: int, gather_first: int, shards, unit_fulls,
                            stream=None) -> None:
    """grads: one list of N grads per stepped unit (1 or 2 units from
    first_unit); shards: one list of N shards per gathered unit (0 to 2 units
    from gather_first), unit_fulls: one destination per gathered unit."""
    flat_g = [p for row in grads for p in row]
    flat_s = [p for row in shards for p in row]
    _check(_L.zero3_step_units_gather(_h(ctx), first_unit, len(grads), _ptrs(flat_g),
                                      len(flat_g), lr, beta1, beta2, eps, t, gather_first,
                                      len(unit_fulls), _ptrs(flat_s), len(flat_s),
                                      _ptrs(unit_fulls), _stream(stream)))


def zero3_reduce_unit(ctx, unit: int, grads, loss_scale: float = 0.0, stream=None) -> None:
    _check(_L.zero3_reduce_unit(_h(ctx), unit, _ptrs(grads), len(grads), loss_scale,
                                _stream(stream)))


def zero3_gather_group(ctx, first_unit: int, shards, unit_fulls, stream=None) -> None:
    """shards: one list of N shards per unit of the group (or the flat
    unit-major list); unit_fulls: one destination per unit."""
    flat = [p for row in shards for p in row] if shards and isinstance(shards[0], (list, tuple)) \
        else list(shards)
    _check(_L.zero3_gather_group(_h(ctx), first_unit, len(unit_fulls), _ptrs(flat), len(flat),
                                 _ptrs(unit_fulls), _stream(stream)))


def zero3_step_group(ctx, first_unit: int, n_units: int, grads, lr: float, beta1: float,
                     beta2: float, eps: float, t: int, stream=None) -> None:
    """grads: N buffers, rank k's grads of the group's units end to end."""
    _check(_L.zero3_step_group(_h(ctx), first_unit, n_units, _ptrs(grads), len(grads), lr,
                               beta1, beta2, eps, t, _stream(stream)))


def zero3_reduce_group(ctx, first_unit: int, n_units: int, grads, loss_scale: float = 0.0,
                       stream=None) -> None:
    _check(_L.zero3_reduce_group(_h(ctx), first_unit, n_units, _ptrs(grads), len(grads),
                                 loss_scale, _stream(stream)))


# ------------------------------------------------- step without allocation

def zero_step_noalloc(ctx, grads, lr: float, beta1: float, beta2: float, eps: float, t: int,
                      loss_scale: float = 0.0, stream=None) -> None:
    """zero_step with the scratch taken from the library's built-in array
    (for callers that cannot allocate device memory; see include/zero.h)."""
    _check(_L.zero_step_noalloc(_h(ctx), _ptrs(grads), len(grads), lr, beta1, beta2, eps, t,
                                loss_scale, _stream(stream)))
