"""zero_step_noalloc: the step for callers that cannot allocate device
memory (the library supplies the scratch from a built-in 16 MiB array).

Checked two ways on the same inputs, two or more calls in a row:
  - against the allocating entry point (zero_step with a bound g_scratch),
    with the tolerances of the other parity tests: master, m, v within
    2e-6*|x| + 1e-9, params within 1 ulp;
  - against the oracle (tests/refs.OracleRun), bit for bit, skip decisions
    included, in the forms the header promises: one state set, a second
    state set bound (the call then updates the current set in place; 16-byte
    and 4-byte aligned sets), and a bound device scalar block.
Self-contained, so it passes alone in a fresh process as well as after the
rest of the suite.
"""
import numpy as np
import pytest
import torch

import synth
import workloads as W
import zero_sharded_optimizer_step_gb300 as z
from tests import refs
from tests.test_gpu_parity import compare_runner

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _close_state(a: torch.Tensor, b: torch.Tensor, what: str):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    ok = (np.abs(a - b) <= 2e-6 * np.abs(b) + 1e-9) | (a == b)
    assert ok.all(), "%s: %d elements out of tolerance" % (what, (~ok).sum())


def _close_params(a: torch.Tensor, b: torch.Tensor, what: str):
    ai = a.view(torch.int16).cpu().numpy().astype(np.int32)
    bi = b.view(torch.int16).cpu().numpy().astype(np.int32)
    ok = (np.abs(ai - bi) <= 1) & ((ai < 0) == (bi < 0))
    assert ok.all(), "%s: %d params more than 1 ulp apart" % (what, (~ok).sum())


class Side:
    """One context with its own state; grads are shared."""

    def __init__(self, numel, world, rank, with_scratch):
        self.ctx = z.zero_init(numel, world, 2, z.ZERO_F16, z.ZERO_F16, rank)
        n = z.zero_ctx_state_elems(self.ctx)
        P = z.zero_ctx_param_elems(self.ctx)
        self.master = torch.zeros(n, device=DEV)
        S = z.zero_ctx_shard_size(self.ctx, -1)
        lo = 0 if rank < 0 else rank * S
        nv = numel if rank < 0 else max(0, min(S, numel - lo))
        synth.fill_device(self.master.data_ptr(), nv, synth.F32, synth.key(3, synth.KIND_MASTER),
                          0.01, torch.cuda.current_stream().cuda_stream, index0=lo)
        self.m = torch.zeros(n, device=DEV)
        self.v = torch.zeros(n, device=DEV)
        self.params = torch.zeros(P, dtype=torch.float16, device=DEV)
        self.g = torch.zeros(n, device=DEV) if with_scratch else None
        self.flag = torch.zeros(1, dtype=torch.int64, device=DEV)
        z.zero_bind(self.ctx, self.master, self.m, self.v, self.params, self.g, self.flag)


def _grads(numel, world, rank, it, scale, n_per_rank):
    S = -(-numel // world)
    lo = 0 if rank < 0 else rank * S
    nv = numel if rank < 0 else max(0, min(S, numel - lo))
    out = []
    for k in range(world):
        t = torch.zeros(n_per_rank, dtype=torch.float16, device=DEV)
        synth.fill_device(t.data_ptr(), nv, synth.F16, synth.key(3, synth.KIND_GRAD, it, k),
                          1e-3 * scale, torch.cuda.current_stream().cuda_stream, index0=lo)
        out.append(t)
    return out


@pytest.mark.parametrize("numel,world,rank", [(1_000_003, 8, -1), (3_000_001, 3, 1)])
def test_noalloc_matches_the_allocating_step(numel, world, rank):
    scale = 1024.0
    a = Side(numel, world, rank, with_scratch=True)
    b = Side(numel, world, rank, with_scratch=False)
    n_per_rank = numel if rank < 0 else -(-numel // world)
    for t in (1, 2):                      # two calls in a row
        g = _grads(numel, world, rank, t, scale, n_per_rank)
        z.zero_step(a.ctx, g, 1e-3, 0.9, 0.999, 1e-8, t, loss_scale=scale)
        z.zero_step_noalloc(b.ctx, g, 1e-3, 0.9, 0.999, 1e-8, t, loss_scale=scale)
        assert z.zero_step_status(a.ctx) == z.zero_step_status(b.ctx) == (False, False)
        torch.cuda.synchronize()
        _close_state(b.master, a.master, "master")
        _close_state(b.m, a.m, "m")
        _close_state(b.v, a.v, "v")
        _close_params(b.params, a.params, "params")


def test_noalloc_skips_like_the_allocating_step():
    numel, world, scale = 500_000, 4, 2.0 ** 16
    a = Side(numel, world, -1, with_scratch=True)
    b = Side(numel, world, -1, with_scratch=False)
    for t in (1, 2):
        g = _grads(numel, world, -1, t, scale, numel)
        if t == 2:
            g[1][4321] = float("inf")
        z.zero_step(a.ctx, g, 1e-3, 0.9, 0.999, 1e-8, t, loss_scale=scale)
        z.zero_step_noalloc(b.ctx, g, 1e-3, 0.9, 0.999, 1e-8, t, loss_scale=scale)
        want = (t == 2, t == 2)
        assert z.zero_step_status(a.ctx) == want and z.zero_step_status(b.ctx) == want
    torch.cuda.synchronize()
    _close_state(b.master, a.master, "master")
    _close_params(b.params, a.params, "params")


# ------------------------------------------------- against the oracle


def _noalloc_step(run, it):
    """Iteration `it` of a Runner's workload through zero_step_noalloc."""
    w = run.w
    run.fill_grads(it)
    hp = run._hp(run.t + 1)           # with a bound scalar block: prepared and copied
    z.zero_step_noalloc(run.ctx, run.grads[0], *hp, run.scale, run.stream)
    return run.finish_step()


def _scaled(rank=-1):
    # fp16 grads and params, loss scale 2^12, a +inf in rank 2 at iteration 3
    w = W.Workload("noalloc", 1_000_003, 8, 2, W.F16, W.F16, rank=rank, steps=5,
                   loss_scale=2.0 ** 12, inject=(3, 2))
    if rank >= 0:
        e = synth.pick_index(w.seed, w.numel, step=3, rank=2)
        w = w.replace(rank=e // w.shard)      # the planted value falls in this shard
    return w


@pytest.mark.parametrize("rank", [-1, 0])
def test_noalloc_equals_the_oracle(rank):
    """One state set, no scratch bound: five calls, the third skipped."""
    from workloads.runner import Runner
    w = _scaled(rank)
    run = Runner(w, scratch=False)
    ref = refs.OracleRun(w)
    for it in range(1, w.steps + 1):
        _noalloc_step(run, it)
        ref.step(it)
    torch.cuda.synchronize()
    assert run.skips == ref.skips == [False, False, True, False, False]
    assert run.scale == ref.scale
    compare_runner(run, ref, exact=True, what="noalloc rank %d" % rank)
    run.close()


def test_noalloc_unscaled_equals_the_oracle():
    """No loss scaling (loss_scale <= 0): never skips, bf16, ragged world."""
    from workloads.runner import Runner
    w = W.Workload("noalloc_u", 777_777, 5, 2, W.BF16, W.BF16, steps=3)
    run = Runner(w, scratch=False)
    ref = refs.OracleRun(w)
    for it in range(1, w.steps + 1):
        _noalloc_step(run, it)
        ref.step(it)
    torch.cuda.synchronize()
    compare_runner(run, ref, exact=True, what="noalloc unscaled")
    run.close()


def _bind_offset_shadow(run, float_offset):
    """A second state set whose buffers start `float_offset` floats into their
    allocations (0: 16-byte aligned; 1: only 4-byte aligned)."""
    n = z.zero_ctx_state_elems(run.ctx)
    bufs = [torch.zeros(n + 8, device=run.dev)[float_offset:float_offset + n] for _ in range(3)]
    run.shadow = tuple(bufs)
    run.cur = torch.zeros(1, dtype=torch.int64, device=run.dev)
    z.zero_bind_shadow(run.ctx, *run.shadow, run.cur)


@pytest.mark.parametrize("float_offset", [0, 1])
def test_noalloc_with_a_second_state_set(float_offset):
    """With a second state set bound, zero_step (one pass) and
    zero_step_noalloc alternate: step 1 by zero_step leaves the second set
    current, step 2 by noalloc updates it in place, step 3 (skipped) by
    noalloc, step 4 by zero_step writes the first set, step 5 by noalloc.
    With the set 4-byte aligned only, every launch takes the per-element
    path; either way the result is the oracle's bit for bit."""
    from workloads.runner import Runner
    w = _scaled()
    run = Runner(w, scratch=False)
    _bind_offset_shadow(run, float_offset)
    ref = refs.OracleRun(w)
    current = []
    for it in range(1, w.steps + 1):
        if it in (1, 4):
            run.step(it)
        else:
            _noalloc_step(run, it)
        ref.step(it)
        current.append(z.zero_current_state(run.ctx))
    torch.cuda.synchronize()
    assert run.skips == ref.skips == [False, False, True, False, False]
    # noalloc updates the current set in place; zero_step flips it
    assert current == [1, 1, 1, 0, 0]
    compare_runner(run, ref, exact=True, what="noalloc shadow offset %d" % float_offset)
    run.close()


def test_noalloc_with_a_device_scalar_block():
    """A bound device scalar block (zero_bind_hyper + zero_prepare_step before
    each call): the kernels read the step's scalars from it; the arguments
    the call gets are ignored.  Bit for bit the oracle's."""
    from workloads.runner import Runner
    w = _scaled()
    run = Runner(w, scratch=False, hyper=True)
    ref = refs.OracleRun(w)
    for it in range(1, w.steps + 1):
        _noalloc_step(run, it)
        ref.step(it)
    torch.cuda.synchronize()
    assert run.skips == ref.skips
    compare_runner(run, ref, exact=True, what="noalloc hyper")
    z.zero_bind_hyper(run.ctx, None)
    run.close()


def test_noalloc_rejects_ranges_beyond_the_builtin_scratch():
    numel = (1 << 22) + 1
    s = Side(numel, 1, -1, with_scratch=False)
    before = s.master.clone()
    g = [torch.zeros(numel, dtype=torch.float16, device=DEV)]
    with pytest.raises(z.ZeroError) as ei:
        z.zero_step_noalloc(s.ctx, g, 1e-3, 0.9, 0.999, 1e-8, 1, loss_scale=1024.0)
    assert ei.value.code == z.ZERO_EINVAL
    assert "scratch" in str(ei.value)
    torch.cuda.synchronize()
    assert torch.equal(s.master, before)     # nothing was launched
