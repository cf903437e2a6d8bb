"""zero3_step_unit_gather: a ZeRO-3 backward visit (unit u's update and the
gather of unit u-1) in one call, against the oracle.

Every gathered buffer (forward and backward) and the final state and params
match the oracle bit for bit; the one-call visit equals the two separate
calls; the library refuses a visit whose halves would touch the same memory
(nothing launched); large shards, the lean gather mode, a bound scalar block
and a capped step occupancy take the two-launch form with the same results.
"""
import pytest
import torch

import workloads as W
import zero_sharded_optimizer_step_gb300 as z
from tests import refs
from tests.test_gpu_parity import compare_runner, to_np

pytestmark = pytest.mark.gpu


def _visit_step(run, it, seen=None):
    """One ZeRO-3 step with fused backward visits, recording what every
    gather left in the unit buffer (the buffer is read after each call)."""
    w = run.w
    run.fill_grads(it)
    hp = run._hp(run.t + 1)
    U = len(w.units)
    z.zero3_begin_step_scaled(run.ctx, run.scale)

    def look(u):
        if seen is not None:
            torch.cuda.synchronize()
            seen.append(to_np(run.unit_full[:w.unit_shard(u) * w.world]).copy())
    for u in range(U):
        z.zero3_gather_unit(run.ctx, u, run.shards[u], run.unit_full, run.stream)
        look(u)
    z.zero3_gather_unit(run.ctx, U - 1, run.shards[U - 1], run.unit_full, run.stream)
    look(U - 1)
    for u in reversed(range(1, U)):
        z.zero3_step_unit_gather(run.ctx, u, run.grads[u], *hp, u - 1, run.shards[u - 1],
                                 run.unit_full, run.stream)
        look(u - 1)
    z.zero3_step_unit(run.ctx, 0, run.grads[0], *hp, run.stream)
    if run.shadow is not None:
        z.zero3_end_step(run.ctx, run.stream)
    return run.finish_step()


CASES = [
    # (rank, grad dtype, param dtype, loss-scaled with two state sets)
    (1, W.BF16, W.BF16, False),
    (-1, W.BF16, W.BF16, False),
    (0, W.F16, W.F16, True),
    (-1, W.F16, W.F16, True),
    (2, W.F32, W.BF16, False),
    (3, W.BF16, W.F32, True),
]


@pytest.mark.parametrize("world,rank,scaled", [(1, 0, True), (1, -1, False), (13, 12, True),
                                               (13, -1, False), (64, 63, False)])
def test_visits_at_edge_worlds(world, rank, scaled):
    """One rank (the sum is the identity), an odd world with the last rank
    (whose shards are mostly padding), and 64 ranks (small shards, many
    rows): gathers, state and params bit for bit the oracle's."""
    from workloads.runner import Runner
    units = [50_001, 1_000, 77_777, 64]
    w = W.Workload("visit_e", sum(units), world, 3, W.BF16, W.BF16, rank=rank, units=units,
                   steps=2, loss_scale=2.0 ** 8 if scaled else 0.0)
    run = Runner(w, shadow=scaled)
    ref = refs.OracleRun(w)
    for it in range(1, w.steps + 1):
        seen = []
        _visit_step(run, it, seen)
        ref.step(it)
        want = [g[2] for g in ref.gathers[-2 * len(units):]]
        for a, b in zip(seen, want):
            assert a.tobytes() == b.tobytes()
    assert run.skips == ref.skips
    compare_runner(run, ref, what="visits world %d rank %d" % (world, rank))
    run.close()


@pytest.mark.parametrize("rank,gdt,pdt,scaled", CASES)
def test_visits_equal_the_oracle(rank, gdt, pdt, scaled):
    """Units of uneven sizes (an empty one and a 7-element one among them),
    4 ranks; loss-scaled cases plant a +inf at iteration 2 (every unit's
    update is discarded and the params recast)."""
    from workloads.runner import Runner
    units = [100_003, 7, 0, 250_000, 33_333, 4096]
    w = W.Workload("visit", sum(units), 4, 3, gdt, pdt, rank=rank, units=units, steps=3,
                   loss_scale=2.0 ** 10 if scaled else 0.0, inject=(2, 1) if scaled else None)
    run = Runner(w, shadow=scaled)
    ref = refs.OracleRun(w)
    for it in range(1, w.steps + 1):
        seen = []
        _visit_step(run, it, seen)
        ref.step(it)
        want = [g[2] for g in ref.gathers[-2 * len(units):]]
        assert len(seen) == len(want)
        for a, b in zip(seen, want):
            assert a.tobytes() == b.tobytes()
    assert run.skips == ref.skips
    if scaled and rank < 0:
        assert ref.skips == [False, True, False]
    compare_runner(run, ref, what="visits %s" % ((rank, gdt, pdt, scaled),))
    run.close()


@pytest.mark.parametrize("mode", ["lean", "hyper", "capped", "large"])
def test_two_launch_forms_equal_the_oracle(mode):
    """The forms in which the call makes the two separate launches."""
    from workloads.runner import Runner
    if mode == "large":
        # shards of 32 MiB and more take the row placement: 16,777,216 bf16
        # elements per shard, then a small unit
        units = [4 * (1 << 24) + 12, 60_000]
        rank = 1
    else:
        units = [200_000, 33_333, 120_000]
        rank = 0
    w = W.Workload("visit2", sum(units), 4, 3, W.BF16, W.BF16, rank=rank, units=units,
                   steps=2)
    run = Runner(w, hyper=mode == "hyper")
    if mode == "lean":
        z.zero_set_gather_mode(run.ctx, z.ZERO_GATHER_LEAN)
    if mode == "capped":
        z.zero_set_step_occupancy(run.ctx, 2)
    ref = refs.OracleRun(w)
    for it in range(1, w.steps + 1):
        seen = []
        _visit_step(run, it, seen if mode != "large" else None)
        ref.step(it)
        if mode != "large":
            want = [g[2] for g in ref.gathers[-2 * len(units):]]
            for a, b in zip(seen, want):
                assert a.tobytes() == b.tobytes()
    torch.cuda.synchronize()
    compare_runner(run, ref, what="visit two launches %s" % mode)
    if mode == "large":
        # the last gather placed unit 0's shards
        S0 = w.unit_shard(0)
        full = to_np(run.unit_full[:S0 * w.world])
        want = ref.gathers[-1][2]
        assert full.tobytes() == want.tobytes()
    if mode == "hyper":
        z.zero_bind_hyper(run.ctx, None)
    run.close()


def test_fused_visits_equal_separate_calls():
    """The Runner's backward forms on one workload: unit-by-unit visits,
    separate calls and (the default for small units) chunks of two --
    identical bits."""
    from workloads.runner import Runner
    units = [300_001, 150_000, 77_777, 500_000]
    w = W.Workload("visit3", sum(units), 8, 3, W.F16, W.F16, rank=5, units=units, steps=3,
                   loss_scale=2.0 ** 12, inject=(2, 3))
    a = Runner(w, shadow=True, visits="fused", fwd_pairs=False)
    b = Runner(w, shadow=True, visits="separate", fwd_pairs=False)
    c = Runner(w, shadow=True)
    assert a.bwd_chunks() is None and c.bwd_chunks() is not None
    for it in range(1, w.steps + 1):
        for r in (a, b, c):
            r.step(it)
    torch.cuda.synchronize()
    assert a.skips == b.skips == c.skips
    for r in (a, c):
        for x, y in zip(r.state(), b.state()):
            assert torch.equal(x, y)
        assert torch.equal(r.params, b.params)
    assert torch.equal(a.unit_full, b.unit_full)
    # unit 0 is gathered last in every form; the chunks leave it in the
    # first unit buffer too (what lies past it differs: another unit's rest)
    n0 = w.unit_shard(0) * w.world
    assert torch.equal(c.unit_full[:n0], b.unit_full[:n0])
    for r in (a, b, c):
        r.close()


def test_visits_that_would_overlap_are_refused():
    """A unit buffer that overlaps the stepped unit's params, state or grads,
    shards that overlap its params, or the same unit on both halves: the call
    returns ZERO_EINVAL and launches nothing."""
    from workloads.runner import Runner
    units = [50_000, 40_000, 30_000]
    w = W.Workload("visit4", sum(units), 4, 3, W.BF16, W.BF16, rank=0, units=units, steps=1)
    run = Runner(w)
    run.fill_grads(1)
    z.zero3_begin_step(run.ctx)
    torch.cuda.synchronize()
    before = [t.clone() for t in (run.master, run.m, run.v, run.params, run.unit_full)]
    hp = (w.lr, w.beta1, w.beta2, w.eps, 1)
    off2 = z.zero_ctx_unit_param_offset(run.ctx, 2)
    soff2 = z.zero_ctx_unit_state_offset(run.ctx, 2)
    bad = [
        # unit_full starting inside unit 2's params
        (2, 1, run.shards[1], run.params[off2:]),
        # unit_full ending inside unit 2's master (viewed as bf16)
        (2, 1, run.shards[1], run.master[soff2 - 100:].view(torch.bfloat16)),
        # unit_full over one of unit 2's grad slices
        (2, 1, run.shards[1], run.grads[2][3]),
        # a shard that is unit 2's own params
        (2, 1, [run.params[off2:]] + list(run.shards[1][1:]), run.unit_full),
        # the same unit on both halves
        (1, 1, run.shards[1], run.unit_full),
    ]
    for unit, gu, shards, full in bad:
        with pytest.raises(z.ZeroError) as ei:
            z.zero3_step_unit_gather(run.ctx, unit, run.grads[unit], *hp, gu, shards, full)
        assert ei.value.code == z.ZERO_EINVAL
    torch.cuda.synchronize()
    for x, y in zip(before, (run.master, run.m, run.v, run.params, run.unit_full)):
        assert torch.equal(x, y)
    run.close()


@pytest.mark.parametrize("rank", [1, -1])
def test_visits_with_decoupled_weight_decay(rank):
    """AdamW (weight decay 0.05) through both step bodies of the visit kernel
    (a small unit takes the 4-wide body, a 1.5M-element one the 8-wide
    body): bit for bit the oracle's."""
    from workloads.runner import Runner
    units = [6_000_004, 10_007, 250_000]
    w = W.Workload("visit_wd", sum(units), 4, 3, W.BF16, W.BF16, rank=rank, units=units,
                   steps=3, weight_decay=0.05)
    run = Runner(w)
    ref = refs.OracleRun(w)
    for it in range(1, w.steps + 1):
        seen = []
        _visit_step(run, it, seen)
        ref.step(it)
        want = [g[2] for g in ref.gathers[-2 * len(units):]]
        for a, b in zip(seen, want):
            assert a.tobytes() == b.tobytes()
    compare_runner(run, ref, what="visits AdamW rank %d" % rank)
    run.close()



def _paired_step(run, it, seen):
    """One ZeRO-3 step with the Runner's forward (pairs of units placed into
    the two unit buffers by one call) and fused backward visits, recording
    what each gather left in its buffer."""
    w = run.w
    run.fill_grads(it)
    hp = run._hp(run.t + 1)
    U = len(w.units)
    z.zero3_begin_step_scaled(run.ctx, run.scale)

    def look(buf, u):
        torch.cuda.synchronize()
        seen.append(to_np(buf[:w.unit_shard(u) * w.world]).copy())
    for f, n in run.fwd_runs():
        run.gather_run(f, n, run.stream)
        look(run.unit_full, f)
        if n == 2:
            look(run.unit_full2, f + 1)
    z.zero3_gather_unit(run.ctx, U - 1, run.shards[U - 1], run.unit_full, run.stream)
    look(run.unit_full, U - 1)
    for u in reversed(range(1, U)):
        z.zero3_step_unit_gather(run.ctx, u, run.grads[u], *hp, u - 1, run.shards[u - 1],
                                 run.unit_full, run.stream)
        look(run.unit_full, u - 1)
    z.zero3_step_unit(run.ctx, 0, run.grads[0], *hp, run.stream)
    if run.shadow is not None:
        z.zero3_end_step(run.ctx, run.stream)
    return run.finish_step()


@pytest.mark.parametrize("units,rank,scaled", [
    ([100_003, 7, 0, 250_000, 33_333, 4096], 1, False),     # six units: three pairs
    ([50_001, 1_000, 77_777, 64, 3], -1, True),             # five: two pairs and a single
])
def test_forward_pairs_equal_the_oracle(units, rank, scaled):
    """The forward's gathers in pairs (zero3_gather_group into two unit
    buffers): every gathered buffer, the state and the params bit for bit
    the oracle's, over steps whose updates change what the next forward
    gathers."""
    from workloads.runner import Runner
    w = W.Workload("pairs", sum(units), 4, 3, W.BF16, W.BF16, rank=rank, units=units, steps=3,
                   loss_scale=2.0 ** 10 if scaled else 0.0, inject=(2, 1) if scaled else None)
    run = Runner(w, shadow=scaled)
    assert run.fwd_runs()[0] == (0, 2)
    ref = refs.OracleRun(w)
    for it in range(1, w.steps + 1):
        seen = []
        _paired_step(run, it, seen)
        ref.step(it)
        want = [g[2] for g in ref.gathers[-2 * len(units):]]
        assert len(seen) == len(want)
        for a, b in zip(seen, want):
            assert a.tobytes() == b.tobytes()
    assert run.skips == ref.skips
    compare_runner(run, ref, what="forward pairs")
    run.close()


def _chunked_step(run, it, fwd, bwd):
    """One ZeRO-3 step as the Runner makes it with small units: the forward
    in pairs, the backward in chunks of two (zero3_step_units_gather),
    recording what every gather left in its buffer, per unit."""
    w = run.w
    run.fill_grads(it)
    hp = run._hp(run.t + 1)
    z.zero3_begin_step_scaled(run.ctx, run.scale)
    bufs = [run.unit_full, run.unit_full2]

    def look(into, first, n):
        torch.cuda.synchronize()
        for j in range(n):
            u = first + j
            into[u] = to_np(bufs[j][:w.unit_shard(u) * w.world]).copy()
    for f, n in run.fwd_runs():
        run.gather_run(f, n, run.stream)
        look(fwd, f, n)
    chunks = run.bwd_chunks()
    run.gather_run(chunks[0][0], chunks[0][1], run.stream)
    look(bwd, *chunks[0])
    for c, (f, n) in enumerate(chunks):
        gf, gn = chunks[c + 1] if c + 1 < len(chunks) else (0, 0)
        z.zero3_step_units_gather(run.ctx, f, [run.grads[u] for u in range(f, f + n)], *hp, gf,
                                  [run.shards[u] for u in range(gf, gf + gn)], bufs[:gn],
                                  run.stream)
        look(bwd, gf, gn)
    if run.shadow is not None:
        z.zero3_end_step(run.ctx, run.stream)
    return run.finish_step()


@pytest.mark.parametrize("units,world,rank,gdt,scaled", [
    ([100_003, 7, 0, 250_000, 33_333, 4096], 4, 1, W.BF16, False),   # three chunks
    ([50_001, 1_000, 77_777, 64, 3], 4, -1, W.F16, True),          # an odd unit out
    ([30_000, 30_000, 30_001, 29_999], 8, 7, W.BF16, True),         # the last rank's padding
    ([5_000, 7_000, 6_000], 32, 0, W.F16, False),                   # 64 rows of placement
])
def test_backward_in_chunks_equals_the_oracle(units, world, rank, gdt, scaled):
    """The backward in chunks of two units, each call stepping a chunk and
    gathering the next into the two unit buffers: every gathered buffer of
    every step, the state and the params bit for bit the oracle's."""
    from workloads.runner import Runner
    w = W.Workload("chunks", sum(units), world, 3, gdt, gdt, rank=rank, units=units, steps=3,
                   loss_scale=2.0 ** 10 if scaled else 0.0, inject=(2, 0) if scaled else None)
    run = Runner(w, shadow=scaled)
    assert run.bwd_chunks() is not None
    ref = refs.OracleRun(w)
    for it in range(1, w.steps + 1):
        fwd, bwd = {}, {}
        _chunked_step(run, it, fwd, bwd)
        ref.step(it)
        mine = ref.gathers[-2 * len(units):]
        for kind, u, want in mine:
            got = (fwd if kind == "fwd" else bwd)[u]
            assert got.tobytes() == want.tobytes(), (it, kind, u)
    assert run.skips == ref.skips
    compare_runner(run, ref, what="backward in chunks")
    run.close()


def test_units_visit_refuses_overlaps():
    """zero3_step_units_gather refuses, launching nothing: a gathered unit
    that is also stepped, three units, overlapping unit buffers."""
    from workloads.runner import Runner
    units = [10_000, 10_000, 10_000, 10_000]
    w = W.Workload("refuse", sum(units), 4, 3, W.BF16, W.BF16, rank=0, units=units, steps=1)
    run = Runner(w)
    hp = run._hp(1)
    z.zero3_begin_step_scaled(run.ctx, 0.0)
    bufs = [run.unit_full, run.unit_full2]
    g = [run.grads[2], run.grads[3]]
    for args in ((2, g, 3, [run.shards[3]], bufs[:1]),                   # 3 stepped and gathered
                 (1, [run.grads[1]] * 3, 0, [run.shards[0]], bufs[:1]),  # three stepped units
                 (2, g, 0, run.shards[0:2], [run.unit_full, run.unit_full[8:]])):   # overlap
        with pytest.raises(z.ZeroError) as ei:
            z.zero3_step_units_gather(run.ctx, args[0], args[1], *hp, args[2], args[3], args[4])
        assert ei.value.code == z.ZERO_EINVAL
    run.close()


@pytest.mark.parametrize("mode", ["lean", "hyper", "capped", "rows"])
def test_units_visit_separate_forms_equal_the_oracle(mode):
    """The forms in which zero3_step_units_gather makes the separate calls'
    launches (the lean gather mode, a bound scalar block, a capped step
    occupancy, more than 64 shards to place): every gathered buffer, the
    state and the params still the oracle's."""
    from workloads.runner import Runner
    units = [200_000, 33_333, 120_000, 7_001]
    world, rank = (64, 3) if mode == "rows" else (4, 0)
    w = W.Workload("chunks2", sum(units), world, 3, W.BF16, W.BF16, rank=rank, units=units,
                   steps=2)
    run = Runner(w, hyper=mode == "hyper")
    if mode == "lean":
        z.zero_set_gather_mode(run.ctx, z.ZERO_GATHER_LEAN)
    if mode == "capped":
        z.zero_set_step_occupancy(run.ctx, 2)
    ref = refs.OracleRun(w)
    for it in range(1, w.steps + 1):
        fwd, bwd = {}, {}
        _chunked_step(run, it, fwd, bwd)
        ref.step(it)
        for kind, u, want in ref.gathers[-2 * len(units):]:
            got = (fwd if kind == "fwd" else bwd)[u]
            assert got.tobytes() == want.tobytes(), (it, kind, u)
    torch.cuda.synchronize()
    compare_runner(run, ref, what="units visit, separate launches: %s" % mode)
    if mode == "hyper":
        z.zero_bind_hyper(run.ctx, None)
    run.close()
