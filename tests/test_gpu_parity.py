"""Parity of the CUDA path (through the C ABI) with the oracle, element by
element, at sizes the oracle finishes in seconds that still span many
thread blocks and end in a ragged tail.

Bars (the method's stated tolerances):
  master, m, v:   |gpu - oracle| <= 2e-6 * |oracle| + 1e-9
  params:         at most 1 ulp apart (16-bit patterns)
  layout, padding, placement, skip decisions: bit-exact
The kernels perform the oracle's operations in the oracle's order, so they
are also expected to be bit-identical; test_bit_identical checks that.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import workloads as W
from tests import refs

pytestmark = pytest.mark.gpu

STORAGE = oracle.NP_STORAGE


def to_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach().contiguous().cpu()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def assert_state_close(got, ref, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    both_nan = np.isnan(got) & np.isnan(ref)
    with np.errstate(invalid="ignore"):
        d = np.abs(got - ref)
        ok = (d <= 2e-6 * np.abs(ref) + 1e-9) | both_nan | (got == ref)
    if not ok.all():
        i = np.flatnonzero(~ok)[:5]
        raise AssertionError("%s: %d elements out of tolerance, e.g. %s: gpu %s oracle %s"
                             % (what, (~ok).sum(), i, got[i], ref[i]))


def assert_params_close(got, ref, dtype, what):
    if dtype == oracle.F32:
        return assert_state_close(got, ref, what)
    g = got.astype(np.int32)
    r = ref.astype(np.int32)
    gv = oracle.widen(got, dtype)
    rv = oracle.widen(ref, dtype)
    nan = np.isnan(gv) & np.isnan(rv)
    # same sign: 1 ulp = adjacent patterns; +0/-0 count as equal
    ok = (np.abs(g - r) <= 1) & ((g >> 15) == (r >> 15)) | nan | (gv == rv)
    if not ok.all():
        i = np.flatnonzero(~ok)[:5]
        raise AssertionError("%s: %d params more than 1 ulp off, e.g. %s" % (what, (~ok).sum(), i))


def assert_bit_identical(got, ref, dtype, what):
    """Equal bit patterns, except that any two NaNs count as equal (their
    payloads depend on the hardware that produced them)."""
    if got.tobytes() == ref.tobytes():
        return
    nan = np.isnan(oracle.widen(got, dtype) if dtype != oracle.F32 else got) & \
        np.isnan(oracle.widen(ref, dtype) if dtype != oracle.F32 else ref)
    diff = (got.view(np.uint32 if dtype == oracle.F32 else np.uint16)
            != ref.view(np.uint32 if dtype == oracle.F32 else np.uint16)) & ~nan
    assert not diff.any(), "%s not bit-identical at %d elements, e.g. %s" % (
        what, diff.sum(), np.flatnonzero(diff)[:5])


def compare_runner(run, ref, exact=True, what=""):
    w = run.w
    if w.stage < 3:
        x, m, v = ref.state[0]
        full_ref = ref.full
    else:
        x = np.concatenate([ref.state[u][0] for u in sorted(ref.state)])
        m = np.concatenate([ref.state[u][1] for u in sorted(ref.state)])
        v = np.concatenate([ref.state[u][2] for u in sorted(ref.state)])
        full_ref = np.concatenate([ref.own[u] for u in sorted(ref.own)])
    cx, cm, cv = run.state()
    gx, gm, gv, gp = to_np(cx), to_np(cm), to_np(cv), to_np(run.params)
    assert_state_close(gx, x, what + " master")
    assert_state_close(gm, m, what + " m")
    assert_state_close(gv, v, what + " v")
    assert_params_close(gp, full_ref, w.param_dtype, what + " params")
    if exact:
        for name, a, b in [("master", gx, x), ("m", gm, m), ("v", gv, v), ("params", gp, full_ref)]:
            assert_bit_identical(a, b, w.param_dtype if name == "params" else oracle.F32,
                                 "%s %s" % (what, name))


def run_both(w, iters=None, shadow=False, hyper=False):
    from workloads.runner import Runner
    iters = iters or list(range(1, w.steps + 1))
    run = Runner(w, shadow=shadow, hyper=hyper)
    ref = refs.OracleRun(w)
    for it in iters:
        run.step(it)
        ref.step(it)
    torch.cuda.synchronize()
    assert run.skips == ref.skips
    return run, ref


def test_bit_identical_tiny_config():
    """The tiny MLP config: 4 ranks, fp32, 3 steps."""
    run, ref = run_both(W.tiny())
    compare_runner(run, ref, exact=True, what="tiny")
    # and the same as plain Adam over the whole vector on the mean grad
    w = W.tiny()
    x = refs.host_master(w)
    m, v = np.zeros_like(x), np.zeros_like(x)
    for t in range(1, 4):
        g = oracle.all_reduce_mean(refs.host_grads(w, t, 0.0), w.grad_dtype, w.numel)
        oracle.adam(x, m, v, g, w.lr, w.beta1, w.beta2, w.eps, t)
    assert to_np(run.master).tobytes() == x.tobytes()
    run.close()


CASES = []
for gdt, pdt in [(W.BF16, W.BF16), (W.F16, W.F16), (W.F32, W.F32), (W.BF16, W.F32),
                 (W.F32, W.BF16), (W.F16, W.BF16), (W.BF16, W.F16), (W.F32, W.F16),
                 (W.F16, W.F32)]:
    CASES.append((1_000_003, 8, gdt, pdt, -1))
for numel, world, rank in [(1_000_003, 3, -1), (1_000_003, 3, 0), (1_000_003, 3, 2),
                           (777_777, 16, 5), (777_777, 16, 15), (500_000, 1, -1),
                           (500_000, 1, 0), (99_999, 64, -1), (99_999, 64, 63),
                           (2_000_001, 13, 7), (100_007, 256, -1), (100_007, 256, 255)]:
    CASES.append((numel, world, W.BF16, W.BF16, rank))
    CASES.append((numel, world, W.F16, W.F32, rank))


@pytest.mark.parametrize("numel,world,gdt,pdt,rank", CASES)
def test_parity_fused(numel, world, gdt, pdt, rank):
    w = W.Workload("case", numel, world, 2, gdt, pdt, rank=rank, steps=3, lr=1e-3)
    run, ref = run_both(w)
    compare_runner(run, ref, what=str((numel, world, gdt, pdt, rank)))
    run.close()


@pytest.mark.parametrize("rank", [-1, 0, 11])
def test_parity_loss_scaled_skip_sequence(rank):
    """Sixteen fp16 ranks, loss scale 2^16, a +inf in rank 5 at iteration 3:
    iterations 1-2 apply, 3 is skipped (nothing written, scale halved), 4-6
    apply with t = 3, 4, 5 -- bit-identical to the oracle."""
    w = W.Workload("scaled", 1_234_567, 16, 2, W.F16, W.F16, rank=rank, steps=6,
                   loss_scale=2.0 ** 16, inject=(3, 5))
    if rank >= 0:
        # the injected element must fall in this rank's shard for a local verdict
        e = synth.pick_index(w.seed, w.numel, step=3, rank=5)
        w = w.replace(rank=e // w.shard)
    run, ref = run_both(w)
    assert ref.skips == [False, False, True, False, False, False]
    assert run.scale == ref.scale == 2.0 ** 15
    compare_runner(run, ref, what="scaled")
    run.close()


def test_two_pass_equals_fused():
    """zero_step_reduce (no scaling) + zero_step_apply == the fused step."""
    import zero_sharded_optimizer_step_gb300 as z
    from workloads.runner import Runner
    w = W.Workload("tp", 654_321, 8, 2, W.BF16, W.BF16, steps=3)
    a = Runner(w)
    b = Runner(w, scratch=True)
    for it in range(1, 4):
        a.fill_grads(it)
        a.launch_step()
        a.finish_step()
        b.fill_grads(it)
        z.zero_step_reduce(b.ctx, b.grads[0], 0.0, b.stream)
        z.zero_step_apply(b.ctx, w.lr, w.beta1, w.beta2, w.eps, it, b.stream)
    torch.cuda.synchronize()
    for x, y in [(a.master, b.master), (a.m, b.m), (a.v, b.v), (a.params, b.params)]:
        assert torch.equal(x, y)


def test_misaligned_buffers_take_the_exact_path():
    """Buffers that start off a 16-byte boundary (element-aligned views)."""
    import zero_sharded_optimizer_step_gb300 as z
    numel, world = 100_003, 5
    w = W.Workload("mis", numel, world, 2, W.BF16, W.BF16, steps=2)
    ref = refs.OracleRun(w)
    P = w.shard * world
    dev = torch.device("cuda:0")
    big = lambda n, dt, off: torch.zeros(n + 16, dtype=dt, device=dev)[off:off + n]  # noqa
    master = big(P, torch.float32, 1)
    m, v = big(P, torch.float32, 3), big(P, torch.float32, 2)
    params = big(P, torch.bfloat16, 5)
    flag = torch.zeros(1, dtype=torch.int64, device=dev)
    master[:] = torch.from_numpy(refs.host_master(w)).to(dev)
    ctx = z.zero_init(numel, world, 2, z.ZERO_BF16, z.ZERO_BF16, -1)
    z.zero_bind(ctx, master, m, v, params, None, flag)
    for t in (1, 2):
        hg = refs.host_grads(w, t, 0.0)
        gd = [big(numel, torch.bfloat16, 1 + k) for k in range(world)]
        for k in range(world):
            gd[k].copy_(torch.from_numpy(hg[k].view(np.int16)).view(torch.bfloat16))
        z.zero_step(ctx, gd, w.lr, w.beta1, w.beta2, w.eps, t)
        ref.step(t)
    torch.cuda.synchronize()
    x, mm, vv = ref.state[0]
    assert to_np(master).tobytes() == x.tobytes()
    assert to_np(m).tobytes() == mm.tobytes() and to_np(v).tobytes() == vv.tobytes()
    assert to_np(params).tobytes() == ref.full.tobytes()


@pytest.mark.parametrize("gdt,offs,poff,mode", [
    # every grad 8 bytes past a 16-byte boundary (a rank's slices of flat
    # vectors at a shard length of 4 mod 8): the grads read in 8-byte halves
    (W.F16, [4, 4, 4, 4, 4], 0, "plain"),
    (W.F16, [4, 4, 4, 4, 4], 4, "shadow"),      # params there too; two state sets, a skip
    (W.BF16, [4, 4, 4, 4, 4], 1, "scratch"),    # the two passes, a skip
    (W.BF16, [4, 4, 4, 4, 4], 0, "avg"),        # stage 1: the mean written too
    (W.BF16, [0, 4, 0, 4, 8], 0, "plain"),      # mixed offsets
    (W.F16, [0, 4, 0, 12, 8], 4, "shadow"),
    (W.F32, [2, 2, 2, 2, 2], 0, "plain"),       # fp32 grads 8 bytes off
    (W.F16, [2, 2, 2, 2, 2], 0, "plain"),       # 4 bytes off: the per-element path
    (W.F16, [0, 0, 0, 0, 0], 4, "shadow"),      # aligned grads, params 8 bytes off
])
def test_grad_offsets_pick_a_load_width(gdt, offs, poff, mode):
    """Rank grads that start off a 16-byte boundary -- a rank's slices of
    flat vectors whose shard length is not a multiple of 8 elements -- read
    the way their offsets allow (8-byte halves, or element by element);
    every result bit-identical to the oracle's, skipped step included."""
    import zero_sharded_optimizer_step_gb300 as z
    numel, world = 100_003, len(offs)
    pdt = W.F16 if gdt == W.F16 else W.BF16
    scaled = mode in ("shadow", "scratch")
    w = W.Workload("offs", numel, world, 1 if mode == "avg" else 2, gdt, pdt, steps=3,
                   loss_scale=2.0 ** 12 if scaled else 0.0, inject=(2, 1) if scaled else None)
    ref = refs.OracleRun(w)
    P = w.shard * world
    dev = torch.device("cuda:0")
    tdt = {W.F32: torch.float32, W.BF16: torch.bfloat16, W.F16: torch.float16}

    def buf(n, dt, off):
        return torch.zeros(n + 16, dtype=dt, device=dev)[off:off + n]

    def dev_copy(a, dt):
        h = torch.from_numpy(a if a.dtype == np.float32 else a.view(np.int16))
        return h.view(tdt[dt]).to(dev)

    f32 = lambda: torch.zeros(P, dtype=torch.float32, device=dev)  # noqa: E731
    master, m, v = f32(), f32(), f32()
    master.copy_(torch.from_numpy(refs.host_master(w)).to(dev))
    params = buf(P, tdt[pdt], poff)
    params.copy_(dev_copy(ref.full, pdt))
    flag = torch.zeros(1, dtype=torch.int64, device=dev)
    scratch = f32() if mode == "scratch" else None
    ctx = z.zero_init(numel, world, w.stage, gdt, pdt, -1)
    z.zero_bind(ctx, master, m, v, params, scratch, flag)
    shadow = None
    if mode == "shadow":
        shadow = (f32(), f32(), f32())
        cur_word = torch.zeros(1, dtype=torch.int64, device=dev)   # held while ctx lives
        z.zero_bind_shadow(ctx, *shadow, cur_word)
    avg = None
    if mode == "avg":
        avg = buf(P, tdt[gdt], 4)
        z.zero_bind_allreduce_out(ctx, avg)
    scale, good, t = w.loss_scale, 0, 0
    for it in (1, 2, 3):
        hg = refs.host_grads(w, it, scale)
        gd = [buf(numel, tdt[gdt], offs[k]) for k in range(world)]
        for k in range(world):
            gd[k].copy_(dev_copy(hg[k], gdt))
        z.zero_step(ctx, gd, w.lr, w.beta1, w.beta2, w.eps, t + 1, scale)
        _, skipped = z.zero_step_status(ctx)
        assert skipped == ref.step(it), it
        if not skipped:
            t += 1
        if scale > 0:
            scale, good = z.zero_scale_update(scale, skipped, good, w.growth_interval)
    torch.cuda.synchronize()
    assert ref.skips == [False, scaled, False]
    cur = (master, m, v) if shadow is None or z.zero_current_state(ctx) == 0 else shadow
    x, mm, vv = ref.state[0]
    for got, want, what in ((cur[0], x, "master"), (cur[1], mm, "m"), (cur[2], vv, "v")):
        assert_bit_identical(to_np(got), want, oracle.F32, what)
    assert_bit_identical(to_np(params), ref.full, pdt, "params")
    if avg is not None:
        want = oracle.cast(oracle.all_reduce_mean(hg, gdt, numel), gdt)
        assert to_np(avg).tobytes() == want.tobytes()
    ctx.close()


@pytest.mark.parametrize("numel,bucket,shadow", [
    (100_000, 0, True),          # S = 20,000: aligned pieces, one pass
    (100_003, 7_777, True),      # S = 20,001: 2-byte-aligned pieces, buckets across shards
    (100_012, 9_000, False),     # S = 20,003 (pieces 8 bytes off for odd ranks), the scratch
])
def test_view_of_several_ranks_equals_the_oracle(numel, bucket, shadow):
    """A view of ranks 1..3 of 5 (zero_init_ranks): the pieces [S, 4S) of
    every rank's gradient stepped in one pass (or bucket by bucket), the
    three shards' state and their places in the full parameter buffer
    bit-identical to the oracle's all-ranks step over the same range, the
    rest of the buffer untouched; a +inf inside the range skips step 2."""
    import zero_sharded_optimizer_step_gb300 as z
    world, first, k = 5, 1, 3
    dt = W.BF16
    w = W.Workload("view", numel, world, 2, dt, dt, steps=3, loss_scale=2.0 ** 10)
    S = w.shard
    P = S * world
    lo, hi = first * S, (first + k) * S
    dev = torch.device("cuda:0")
    x = refs.host_master(w)
    m_ref, v_ref = np.zeros(P, np.float32), np.zeros(P, np.float32)
    full_ref = oracle.cast(x, dt)
    full0 = full_ref.copy()
    ctx = z.zero_init_ranks(numel, world, 2, dt, dt, first, k)
    assert z.zero_ctx_state_elems(ctx) == k * S
    f32 = lambda: torch.zeros(k * S, dtype=torch.float32, device=dev)  # noqa: E731
    master, m, v = f32(), f32(), f32()
    master.copy_(torch.from_numpy(x[lo:hi]).to(dev))
    params = torch.from_numpy(full_ref.view(np.int16)).to(dev).view(torch.bfloat16)
    flag = torch.zeros(1, dtype=torch.int64, device=dev)
    scratch = None if shadow else f32()
    z.zero_bind(ctx, master, m, v, params, scratch, flag)
    if shadow:
        sets = (f32(), f32(), f32())
        cur_word = torch.zeros(1, dtype=torch.int64, device=dev)
        z.zero_bind_shadow(ctx, *sets, cur_word)
    scale, good, t = w.loss_scale, 0, 0
    for it in (1, 2, 3):
        hg = refs.host_grads(w, it, scale)
        if it == 2:
            hg[3][lo + 12_345] = oracle.cast(np.array([np.inf], np.float32), dt)[0]
        skipped_ref, _ = oracle.zero_step(hg, dt, numel, x, m_ref, v_ref, full_ref, dt, w.lr,
                                          w.beta1, w.beta2, w.eps, t + 1, loss_scale=scale)
        full_g = []
        for g in hg:
            d = torch.zeros(P, dtype=torch.bfloat16, device=dev)
            d[:numel].copy_(torch.from_numpy(g.view(np.int16)).view(torch.bfloat16))
            full_g.append(d)
        pieces = [d[lo:hi] for d in full_g]
        if bucket:
            z.zero_bucket_begin(ctx, scale)
            for off in range(0, k * S, bucket):
                cnt = min(bucket, k * S - off)
                z.zero_bucket_step(ctx, off, cnt, [pc[off:off + cnt] for pc in pieces], w.lr,
                                   w.beta1, w.beta2, w.eps, t + 1)
            z.zero_bucket_end(ctx, w.lr, w.beta1, w.beta2, w.eps, t + 1)
        else:
            z.zero_step(ctx, pieces, w.lr, w.beta1, w.beta2, w.eps, t + 1, scale)
        _, skipped = z.zero_step_status(ctx)
        assert skipped == bool(skipped_ref) == (it == 2), it
        if not skipped:
            t += 1
        scale, good = z.zero_scale_update(scale, skipped, good, w.growth_interval)
    torch.cuda.synchronize()
    cur = (master, m, v) if not shadow or z.zero_current_state(ctx) == 0 else sets
    for got, want, what in ((cur[0], x, "master"), (cur[1], m_ref, "m"), (cur[2], v_ref, "v")):
        assert_bit_identical(to_np(got), want[lo:hi], oracle.F32, what)
    got = to_np(params)
    assert_bit_identical(got[lo:hi], full_ref[lo:hi], dt, "params in the view's range")
    assert got[:lo].tobytes() == full0[:lo].tobytes()
    assert got[hi:].tobytes() == full0[hi:].tobytes()
    ctx.close()


@pytest.mark.parametrize("rank", [-1, 2])
def test_stage1_allreduce_output(rank):
    """Stage 1 keeps the full averaged grads: RS + AG == AR, bit-exact."""
    import zero_sharded_optimizer_step_gb300 as z
    from workloads.runner import Runner
    w = W.Workload("s1", 300_007, 6, 1, W.BF16, W.BF16, rank=rank, steps=1)
    run = Runner(w)
    avg = torch.zeros(w.shard * w.world, dtype=torch.bfloat16, device="cuda:0")
    z.zero_bind_allreduce_out(run.ctx, avg)
    run.step(1)
    torch.cuda.synchronize()
    want = oracle.cast(oracle.all_reduce_mean(refs.host_grads(w, 1, 0.0), w.grad_dtype,
                                              w.numel), w.grad_dtype)
    got = to_np(avg)
    if rank < 0:
        assert got.tobytes() == want.tobytes()
    else:
        S = w.shard
        assert got[rank * S:(rank + 1) * S].tobytes() == want[rank * S:(rank + 1) * S].tobytes()
        assert not got[:rank * S].any() and not got[(rank + 1) * S:].any()
    run.close()


@pytest.mark.parametrize("S,world,dtype,dst_off", [(1, 1, W.BF16, 0), (7, 3, W.BF16, 1),
                                                    (1001, 8, W.F16, 3), (4096, 4, W.F32, 1),
                                                    (117_187, 64, W.BF16, 0),
                                                    (250_001, 5, W.BF16, 7),
                                                    (3_000_000, 4, W.F32, 2)])
def test_gather_placement(S, world, dtype, dst_off):
    """All-gather placement is a bit-exact copy for any alignment."""
    import zero_sharded_optimizer_step_gb300 as z
    dev = torch.device("cuda:0")
    tdt = {W.F32: torch.float32, W.BF16: torch.bfloat16, W.F16: torch.float16}[dtype]
    numel = S * world
    ctx = z.zero_init(numel, world, 2, dtype, dtype, 0)
    shards_h = [synth.fill_host(S, dtype, synth.key(5, W.KIND_SHARD, 0, k), 1.0)
                for k in range(world)]
    shards = []
    for k, h in enumerate(shards_h):
        buf = torch.zeros(S + 16, dtype=tdt, device=dev)[(k * 3) % 8:][:S]
        src = torch.from_numpy(h.view(np.int16) if dtype != W.F32 else h)
        buf.copy_(src.view(tdt) if dtype != W.F32 else src)
        shards.append(buf)
    full = torch.full((numel + 16,), 7, dtype=tdt, device=dev)[dst_off:dst_off + numel]
    master = torch.zeros(S, device=dev)
    flag = torch.zeros(1, dtype=torch.int64, device=dev)
    z.zero_bind(ctx, master, master, master, full, None, flag)
    skip = world // 2
    z.zero_allgather(ctx, [s if k != skip else None for k, s in enumerate(shards)], full, dtype)
    torch.cuda.synchronize()
    got = to_np(full)
    want = oracle.all_gather(shards_h, dtype)
    keep = np.ones(numel, bool)
    keep[skip * S:(skip + 1) * S] = False
    assert got[keep].tobytes() == want[keep].tobytes()
    seven = to_np(torch.full((1,), 7, dtype=tdt))
    assert (got[~keep] == seven[0]).all()      # the skipped shard is untouched


@pytest.mark.parametrize("rank,scaled", [(1, False), (-1, False), (0, True)])
def test_stage3_units(rank, scaled):
    """ZeRO-3: per unit, gather before forward and before backward, then the
    unit's reduce + Adam; every gathered buffer and the final state match."""
    import zero_sharded_optimizer_step_gb300 as z
    from workloads.runner import Runner
    units = [100_003, 7, 250_000, 33_333]
    w = W.Workload("z3", sum(units), 4, 3, W.BF16, W.BF16, rank=rank, units=units, steps=3,
                   loss_scale=2.0 ** 10 if scaled else 0.0)
    run = Runner(w)
    ref = refs.OracleRun(w)
    for it in range(1, 4):
        run.fill_grads(it)
        t = run.t + 1
        z.zero3_begin_step(run.ctx)
        seen = []
        for u in range(len(units)):
            z.zero3_gather_unit(run.ctx, u, run.shards[u], run.unit_full)
            seen.append(to_np(run.unit_full[:w.unit_shard(u) * w.world]))
        for u in reversed(range(len(units))):
            z.zero3_gather_unit(run.ctx, u, run.shards[u], run.unit_full)
            seen.append(to_np(run.unit_full[:w.unit_shard(u) * w.world]))
            if scaled:
                z.zero3_reduce_unit(run.ctx, u, run.grads[u], run.scale)
            else:
                z.zero3_step_unit(run.ctx, u, run.grads[u], w.lr, w.beta1, w.beta2, w.eps, t)
        if scaled:
            z.zero_step_apply(run.ctx, w.lr, w.beta1, w.beta2, w.eps, t)
        run.finish_step()
        ref.step(it)
        want = [g[2] for g in ref.gathers[-2 * len(units):]]
        for a, b in zip(seen, want):
            assert a.tobytes() == b.tobytes()
    assert run.skips == ref.skips
    compare_runner(run, ref, what="stage3")
    run.close()


def test_degenerate_sizes():
    """numel = 0 (nothing to do), numel < world (ranks owning only padding)
    and world = 1 (the identity reduce)."""
    import zero_sharded_optimizer_step_gb300 as z
    from workloads.runner import Runner
    c = z.zero_init(0, 8, 2, z.ZERO_BF16, z.ZERO_BF16, -1)
    dev = torch.device("cuda:0")
    e = torch.zeros(0, device=dev)
    flag = torch.zeros(1, dtype=torch.int64, device=dev)
    z.zero_bind(c, e, e, e, e, None, flag)
    z.zero_step(c, [None] * 8, 1e-3, 0.9, 0.999, 1e-8, 1)
    assert z.zero_step_status(c) == (False, False)
    for numel, world, rank in [(3, 4, -1), (3, 4, 3), (1, 1, -1), (5, 8, 6), (17, 1, 0)]:
        w = W.Workload("deg", numel, world, 2, W.BF16, W.F32, rank=rank, steps=2)
        run, ref = run_both(w)
        compare_runner(run, ref, what="deg")
        run.close()


def test_nonfinite_without_loss_scaling_is_reported_not_skipped():
    from workloads.runner import Runner
    w = W.Workload("nf", 10_000, 4, 2, W.F32, W.F32, steps=1, inject=(1, 2))
    run, ref = run_both(w)
    assert run.skips == [False]
    compare_runner(run, ref, what="nf")
    import zero_sharded_optimizer_step_gb300 as z
    assert z.zero_step_status(run.ctx) == (True, False)
    run.close()


def test_error_codes_on_device():
    import zero_sharded_optimizer_step_gb300 as z
    dev = torch.device("cuda:0")
    c = z.zero_init(1000, 4, 2, z.ZERO_BF16, z.ZERO_BF16, -1)
    P = z.zero_ctx_state_elems(c)
    f = torch.zeros(P, device=dev)
    p = torch.zeros(P, dtype=torch.bfloat16, device=dev)
    flag = torch.zeros(1, dtype=torch.int64, device=dev)
    z.zero_bind(c, f, f.clone(), f.clone(), p, None, flag)
    g = [torch.zeros(1000, dtype=torch.bfloat16, device=dev) for _ in range(4)]
    cases = [
        (lambda: z.zero_step(c, g[:3], 1e-3, 0.9, 0.999, 1e-8, 1), z.ZERO_EINVAL),
        (lambda: z.zero_step(c, g, 1e-3, 0.9, 0.999, 1e-8, 0), z.ZERO_EINVAL),
        (lambda: z.zero_step(c, g[:3] + [None], 1e-3, 0.9, 0.999, 1e-8, 1), z.ZERO_EINVAL),
        (lambda: z.zero_step(c, g[:3] + [g[3].data_ptr() + 1], 1e-3, 0.9, 0.999, 1e-8, 1),
         z.ZERO_EALIGN),
        (lambda: z.zero_step(c, g, 1e-3, 0.9, 0.999, 1e-8, 1, loss_scale=1024.0),
         z.ZERO_ESTATE),
        (lambda: z.zero3_gather_unit(c, 0, g, p), z.ZERO_EINVAL),
        (lambda: z.zero_bind(c, f.data_ptr() + 2, f, f, p, None, flag), z.ZERO_EALIGN),
        # outside the ranges Adam is defined on (as torch.optim.Adam checks)
        (lambda: z.zero_step(c, g, -1e-3, 0.9, 0.999, 1e-8, 1), z.ZERO_EINVAL),
        (lambda: z.zero_step(c, g, float("nan"), 0.9, 0.999, 1e-8, 1), z.ZERO_EINVAL),
        (lambda: z.zero_step(c, g, 1e-3, 1.0, 0.999, 1e-8, 1), z.ZERO_EINVAL),
        (lambda: z.zero_step(c, g, 1e-3, 0.9, 1.0, 1e-8, 1), z.ZERO_EINVAL),
        (lambda: z.zero_step(c, g, 1e-3, -0.1, 0.999, 1e-8, 1), z.ZERO_EINVAL),
        (lambda: z.zero_step(c, g, 1e-3, 0.9, 0.999, -1e-8, 1), z.ZERO_EINVAL),
        (lambda: z.zero_step(c, g, 1e-3, 0.9, 0.999, float("inf"), 1), z.ZERO_EINVAL),
        (lambda: z.zero_step(c, g, 1e-3, 0.9, 0.999, 1e-8, 1, loss_scale=float("inf")),
         z.ZERO_EINVAL),
        (lambda: z.zero_step(c, g, 1e-3, 0.9, 0.999, 1e-8, 1, loss_scale=float("nan")),
         z.ZERO_EINVAL),
        (lambda: z.zero_bucket_begin(c, float("inf")), z.ZERO_EINVAL),
    ]
    for fn, code in cases:
        with pytest.raises(z.ZeroError) as ei:
            fn()
        assert ei.value.code == code, z.zero_last_error()
    torch.cuda.synchronize()
    assert not f.any()         # nothing was launched


@pytest.mark.parametrize("numel,world,rank", [(1_000_001, 6, 1), (999_999, 64, 63)])
def test_one_rank_step_then_placement(numel, world, rank):
    """One rank's view: its shard is updated in place in the full buffer,
    then the other ranks' shards are placed around it."""
    w = W.Workload("or", numel, world, 2, W.BF16, W.BF16, rank=rank, steps=2,
                   gather_after=True)
    run, ref = run_both(w)
    compare_runner(run, ref, what="one-rank+placement")
    run.close()


# ------------------------------------------- one pass with two state sets

@pytest.mark.parametrize("rank", [-1, 0])
def test_shadow_single_pass_skip_sequence(rank):
    """The loss-scaled step as one pass over two state sets: the skipped
    iteration leaves the old set current and recasts the params from it;
    bit-identical to the oracle over the whole sequence."""
    w = W.Workload("shadow", 1_234_567, 16, 2, W.F16, W.F16, rank=rank, steps=6,
                   loss_scale=2.0 ** 16, inject=(3, 5))
    if rank >= 0:
        e = synth.pick_index(w.seed, w.numel, step=3, rank=5)
        w = w.replace(rank=e // w.shard)
    run, ref = run_both(w, shadow=True)
    assert ref.skips == [False, False, True, False, False, False]
    import zero_sharded_optimizer_step_gb300 as z
    # five applied steps flip the current set five times
    assert z.zero_current_state(run.ctx) == 1
    compare_runner(run, ref, what="shadow")
    run.close()


@pytest.mark.parametrize("numel,world,gdt,pdt,rank", [(1_000_003, 8, W.BF16, W.BF16, -1),
                                                     (1_000_003, 3, W.F16, W.F32, 2),
                                                     (99_999, 64, W.F32, W.BF16, 63)])
def test_shadow_unscaled_steps(numel, world, gdt, pdt, rank):
    w = W.Workload("shadow-u", numel, world, 2, gdt, pdt, rank=rank, steps=3, lr=1e-3)
    run, ref = run_both(w, shadow=True)
    compare_runner(run, ref, what="shadow-u")
    run.close()


def test_shadow_mixed_with_two_pass_steps():
    """With two sets bound, the two-pass calls update the current set in
    place; alternating them with one-pass steps still matches the oracle."""
    import zero_sharded_optimizer_step_gb300 as z
    from workloads.runner import Runner
    w = W.Workload("mix", 500_001, 8, 2, W.BF16, W.BF16, steps=4, loss_scale=2.0 ** 8)
    run = Runner(w, scratch=True, shadow=True)
    ref = refs.OracleRun(w)
    for it in range(1, 5):
        run.fill_grads(it)
        if it % 2:
            run.launch_step()
        else:
            z.zero_step_reduce(run.ctx, run.grads[0], run.scale, run.stream)
            z.zero_step_apply(run.ctx, w.lr, w.beta1, w.beta2, w.eps, run.t + 1, run.stream)
        run.finish_step()
        ref.step(it)
    compare_runner(run, ref, what="mix")
    run.close()


# -------------------------------------------------------------------- AdamW

@pytest.mark.parametrize("shadow,scaled,rank", [(False, False, -1), (False, True, -1),
                                               (True, True, -1), (False, False, 2)])
def test_adamw_parity(shadow, scaled, rank):
    """Decoupled weight decay on every path: fused, two-pass, one pass over
    two state sets, one rank's view -- bit-identical to the oracle."""
    w = W.Workload("adamw", 777_777, 8, 2, W.BF16, W.BF16, rank=rank, steps=3, lr=1e-3,
                   weight_decay=0.1, loss_scale=2.0 ** 10 if scaled else 0.0)
    run, ref = run_both(w, shadow=shadow)
    compare_runner(run, ref, what="adamw")
    run.close()


def test_adamw_stage3_units():
    units = [300_001, 77, 123_456]
    w = W.Workload("adamw3", sum(units), 4, 3, W.F16, W.F16, rank=1, units=units, steps=2,
                   weight_decay=0.01)
    run, ref = run_both(w)
    compare_runner(run, ref, what="adamw3")
    run.close()


def test_weight_decay_argument_checked():
    import zero_sharded_optimizer_step_gb300 as z
    c = z.zero_init(10, 2, 2, z.ZERO_F32, z.ZERO_F32, -1)
    for bad in (-0.1, float("nan"), float("inf")):
        with pytest.raises(z.ZeroError):
            z.zero_set_weight_decay(c, bad)
    z.zero_set_weight_decay(c, 0.0)


# ------------------------------------------------------------ bucketed step

@pytest.mark.parametrize("bucket,shadow,scaled,rank", [
    (100_000, False, False, -1),       # multiples of 8: vector path
    (99_999, False, False, -1),        # ragged buckets: per-element path
    (65_536, True, True, -1),          # one pass over two state sets, with a skip
    (65_536, False, True, -1),         # two passes, with a skip
    (50_000, False, False, 3),         # one rank's view
    (10_000_000, True, True, 0),       # a single bucket larger than the shard
])
def test_bucketed_step_equals_the_whole_step(bucket, shadow, scaled, rank):
    w = W.Workload("bk", 654_321, 8, 2, W.F16, W.F16, rank=rank, steps=4, bucket=bucket,
                   loss_scale=2.0 ** 12 if scaled else 0.0, inject=(2, 5) if scaled else None)
    if scaled and rank >= 0:
        e = synth.pick_index(w.seed, w.numel, step=2, rank=5)
        w = w.replace(rank=e // w.shard)
    run, ref = run_both(w, shadow=shadow)
    if scaled:
        assert ref.skips == [False, True, False, False]
    compare_runner(run, ref, what="bucketed")
    run.close()


def test_bucket_protocol_errors():
    import zero_sharded_optimizer_step_gb300 as z
    from workloads.runner import Runner
    w = W.Workload("bkerr", 1000, 4, 2, W.BF16, W.BF16, steps=1)
    run = Runner(w)
    g = run.grads[0]
    with pytest.raises(z.ZeroError):                       # not begun
        z.zero_bucket_step(run.ctx, 0, 8, g, 1e-3, 0.9, 0.999, 1e-8, 1)
    z.zero_bucket_begin(run.ctx)
    with pytest.raises(z.ZeroError):                       # outside the range
        z.zero_bucket_step(run.ctx, 999, 8, g, 1e-3, 0.9, 0.999, 1e-8, 1)
    with pytest.raises(z.ZeroError):                       # whole step while open
        z.zero_step(run.ctx, g, 1e-3, 0.9, 0.999, 1e-8, 1)
    with pytest.raises(z.ZeroError):                       # twice begun
        z.zero_bucket_begin(run.ctx)
    with pytest.raises(z.ZeroError):                       # apply pass while open
        z.zero_step_apply(run.ctx, 1e-3, 0.9, 0.999, 1e-8, 1)
    with pytest.raises(z.ZeroError):                       # built-in scratch step while open
        z.zero_step_noalloc(run.ctx, g, 1e-3, 0.9, 0.999, 1e-8, 1)
    id_open = z.zero_step_id(run.ctx)
    z.zero_bucket_end(run.ctx, 1e-3, 0.9, 0.999, 1e-8, 1)
    assert z.zero_step_id(run.ctx) == id_open              # the refused calls began no step
    with pytest.raises(z.ZeroError):                       # loss-scaled, no scratch or set
        z.zero_bucket_begin(run.ctx, 1024.0)
    run.close()


# --------------------------------------------------- ZeRO-3 with prefetch

@pytest.mark.parametrize("rank,scaled", [(2, False), (-1, True), (1, True)])
def test_zero3_prefetch_schedule_matches_serial_and_oracle(rank, scaled):
    """Gathers prefetched on a second stream into alternating unit buffers
    leave every result as the serial schedule and the oracle have it; with
    loss scaling (Adam deferred to one apply after the last unit) the step
    with a planted +inf is skipped by every unit."""
    from workloads.runner import Runner
    from workloads.zero3_schedule import Zero3Schedule
    units = [200_003, 150_000, 99_999, 250_000]
    w = W.Workload("z3p", sum(units), 4, 3, W.BF16, W.BF16, rank=rank, units=units, steps=4,
                   loss_scale=2.0 ** 10 if scaled else 0.0, inject=(2, 1) if scaled else None)
    runs = {}
    for mode, steps_bg in (("serial", False), ("overlap", False), ("overlap", True)):
        run = Runner(w)
        sch = Zero3Schedule(run, 2000, 4000, 64, mode, overlap_steps=steps_bg)
        for it in range(1, 5):
            run.fill_grads(it)
            sch.launch_step()
            if scaled:
                run.finish_step()
        torch.cuda.synchronize()
        runs[(mode, steps_bg)] = run
    ref = refs.OracleRun(w)
    for it in range(1, 5):
        ref.step(it)
    serial = runs[("serial", False)]
    for key in [("overlap", False), ("overlap", True)]:
        for a, b in [(serial.master, runs[key].master), (serial.params, runs[key].params)]:
            assert torch.equal(a, b)
    if scaled:
        for run in runs.values():
            assert run.skips == ref.skips
        assert ref.skips == [0, 1, 0, 0]      # the +inf lands in rank 1's part of unit 0
    else:
        for run in runs.values():
            run.skips = ref.skips
    compare_runner(runs[("overlap", False)], ref, what="prefetch")
    compare_runner(runs[("overlap", True)], ref, what="prefetch, steps in the background")


@pytest.mark.parametrize("S,world,dtype,src_off,dst_off", [
    (25_297_920, 8, W.BF16, 0, 0),      # one Llama-7B unit: the TMA path
    (16384 + 8, 5, W.F16, 0, 0),        # ragged last tile (shard of 32,784 bytes)
    (4096, 3, W.F32, 0, 0),
    (1001, 8, W.BF16, 0, 0),            # 2,002-byte shards: not 16-byte multiples -> fallback
    (250_000, 4, W.BF16, 1, 0),         # unaligned sources -> fallback
])
def test_lean_gather_placement(S, world, dtype, src_off, dst_off):
    """The bulk-copy (lean) gather places bit-exactly; gathers it cannot take
    fall back to the SM kernel; no wait runs out."""
    import zero_sharded_optimizer_step_gb300 as z
    dev = torch.device("cuda:0")
    tdt = {W.F32: torch.float32, W.BF16: torch.bfloat16, W.F16: torch.float16}[dtype]
    before = z.zero_gather_timeouts()
    ctx = z.zero_init(S * world, world, 3, dtype, dtype, 0, [S * world])
    z.zero_set_gather_mode(ctx, z.ZERO_GATHER_LEAN)
    hs = [synth.fill_host(S, dtype, synth.key(9, W.KIND_SHARD, 0, k), 1.0) for k in range(world)]
    shards = []
    for h in hs:
        buf = torch.zeros(S + 16, dtype=tdt, device=dev)[src_off:src_off + S]
        src = torch.from_numpy(h.view(np.int16) if dtype != W.F32 else h)
        buf.copy_(src.view(tdt) if dtype != W.F32 else src)
        shards.append(buf)
    full = torch.zeros(S * world + 16, dtype=tdt, device=dev)[dst_off:dst_off + S * world]
    st = torch.zeros(S, device=dev)
    flag = torch.zeros(1, dtype=torch.int64, device=dev)
    params = torch.zeros(S, dtype=tdt, device=dev)      # bound buffers live as long as ctx
    z.zero_bind(ctx, st, st, st, params, None, flag)
    z.zero3_begin_step(ctx)
    for _ in range(2):
        z.zero3_gather_unit(ctx, 0, shards, full)
    torch.cuda.synchronize()
    assert to_np(full).tobytes() == oracle.all_gather(hs, dtype).tobytes()
    assert z.zero_gather_timeouts() == before


def test_lean_gather_wait_that_runs_out_is_reported():
    """The lean gather's bounded waits, made to run out on purpose (a poll
    limit of 0: no fault, no hang): every CTA with work gives up at its
    first tile, drains the loads it issued and places nothing; the counter
    reports it (ZERO_ETIMEOUT); with the default limit restored the same
    context places bit-exactly again."""
    import zero_sharded_optimizer_step_gb300 as z
    dev = torch.device("cuda:0")
    S, world, dtype = 250_000, 4, W.BF16
    hs = [synth.fill_host(S, dtype, synth.key(10, W.KIND_SHARD, 0, k), 1.0) for k in range(world)]
    shards = [torch.from_numpy(h.view(np.int16)).to(dev).view(torch.bfloat16) for h in hs]
    ctx = z.zero_init(S * world, world, 3, dtype, dtype, 0, [S * world])
    z.zero_set_gather_mode(ctx, z.ZERO_GATHER_LEAN)
    st = torch.zeros(S, device=dev)
    params = torch.zeros(S, dtype=torch.bfloat16, device=dev)   # bound buffers live as
    flag = torch.zeros(1, dtype=torch.int64, device=dev)        # long as ctx
    z.zero_bind(ctx, st, st, st, params, None, flag)
    z.zero3_begin_step(ctx)
    full = torch.full((S * world,), 7.0, dtype=torch.bfloat16, device=dev)
    sentinel = to_np(full).tobytes()
    before = z.zero_gather_timeouts()
    try:
        z.zero_set_gather_wait_polls(0)
        z.zero3_gather_unit(ctx, 0, shards, full)
        torch.cuda.synchronize()
        ran_out = z.zero_gather_timeouts() - before
    finally:
        z.zero_set_gather_wait_polls(-1)
    assert ran_out >= 1
    assert to_np(full).tobytes() == sentinel           # nothing was placed
    import ctypes
    from zero_sharded_optimizer_step_gb300 import binding as zb
    c = ctypes.c_uint32(0)
    assert zb._L.zero_gather_timeouts(ctypes.byref(c)) == z.ZERO_ETIMEOUT
    after = z.zero_gather_timeouts()
    z.zero3_gather_unit(ctx, 0, shards, full)
    torch.cuda.synchronize()
    assert to_np(full).tobytes() == oracle.all_gather(hs, dtype).tobytes()
    assert z.zero_gather_timeouts() == after


@pytest.mark.parametrize("shadow,scaled", [(True, True), (False, False), (False, True)])
def test_zero2_buckets_stepped_during_backward(shadow, scaled):
    """The bucketed ZeRO-2 step run during backward (each bucket on a second
    stream while a stand-in kernel plays the next bucket's backward) equals
    the oracle bit for bit, with a planted +inf skipping iteration 2 when
    loss-scaled -- in both loss-scaled forms (two state sets; one set with
    the scratch, where zero_bucket_end applies Adam after the last bucket)."""
    from workloads.runner import Runner
    from workloads.zero2_schedule import Zero2Schedule
    w = W.Workload("z2o", 1_000_003, 8, 2, W.BF16, W.BF16, steps=3, bucket=100_000,
                   loss_scale=2.0 ** 10 if scaled else 0.0, inject=(2, 5) if scaled else None)
    run = Runner(w, shadow=shadow)
    ref = refs.OracleRun(w)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    sch = Zero2Schedule(run, 2000, 4000, 2 * sms, "overlap")
    for it in range(1, w.steps + 1):
        run.fill_grads(it)
        sch.launch_step()
        if scaled:
            run.finish_step()
        else:
            run.skips.append(False)
        ref.step(it)
    torch.cuda.synchronize()
    assert run.skips == ref.skips == ([False, True, False] if scaled else [False] * 3)
    compare_runner(run, ref, what="zero2 overlap")
    run.close()


# -------------------------------------------------- FSDP2's dim-0 layout

@pytest.mark.parametrize("rank,scaled", [(1, False), (-1, False), (3, True), (0, False)])
def test_dim0_layout_units(rank, scaled):
    """Per-parameter units sharded by whole rows (the MLP's four tensors and
    uneven Llama-like shapes): gathers before forward and backward, per-unit
    reduce + Adam, bit-identical to the oracle; ranks past the last row hold
    only padding."""
    import zero_sharded_optimizer_step_gb300 as z
    from workloads.runner import Runner
    shapes = [(256, 64), (256, 1), (10, 256), (10, 1), (4097, 33), (3, 11)]
    w = W.dim0(shapes, 4, rank=rank, steps=3, loss_scale=2.0 ** 8 if scaled else 0.0)
    run = Runner(w)
    ref = refs.OracleRun(w)
    for u, (rows, row) in enumerate(shapes):
        assert z.zero_ctx_shard_size(run.ctx, u) == -(-rows // 4) * row
    for it in range(1, 4):
        run.fill_grads(it)
        t = run.t + 1
        z.zero3_begin_step(run.ctx)
        seen = []
        order = list(range(len(shapes))) + list(reversed(range(len(shapes))))
        for i, u in enumerate(order):
            z.zero3_gather_unit(run.ctx, u, run.shards[u], run.unit_full)
            seen.append(to_np(run.unit_full[:w.unit_shard(u) * w.world]))
            if i >= len(shapes):
                if scaled:
                    z.zero3_reduce_unit(run.ctx, u, run.grads[u], run.scale)
                else:
                    z.zero3_step_unit(run.ctx, u, run.grads[u], w.lr, w.beta1, w.beta2, w.eps, t)
        if scaled:
            z.zero_step_apply(run.ctx, w.lr, w.beta1, w.beta2, w.eps, t)
        run.finish_step()
        ref.step(it)
        want = [g[2] for g in ref.gathers[-2 * len(shapes):]]
        for a, b in zip(seen, want):
            assert a.tobytes() == b.tobytes()
    assert run.skips == ref.skips
    compare_runner(run, ref, what="dim0")
    run.close()


# ------------------------------------------- groups of units (per module)

@pytest.mark.parametrize("rank", [-1, 0, 3])
def test_group_gather_equals_unit_gathers(rank):
    """One launch placing every shard of a run of units equals the per-unit
    gathers byte for byte, padded units and odd row lengths included."""
    import zero_sharded_optimizer_step_gb300 as z
    from workloads.runner import Runner
    shapes = [(256, 64), (10, 1), (4097, 33), (3, 11), (64, 7)]
    w = W.dim0(shapes, 4, rank=rank, steps=1)
    run = Runner(w)
    z.zero3_begin_step(run.ctx)
    want = []
    for u in range(1, 5):
        z.zero3_gather_unit(run.ctx, u, run.shards[u], run.unit_full)
        want.append(to_np(run.unit_full[:w.unit_shard(u) * w.world]).copy())
    from workloads.runner import TORCH_DTYPE
    dt = TORCH_DTYPE[w.param_dtype]
    fulls = [torch.full((w.unit_shard(u) * w.world + 3,), 7.0, dtype=dt,
                        device="cuda:0")[1:1 + w.unit_shard(u) * w.world] for u in range(1, 5)]
    z.zero3_gather_group(run.ctx, 1, run.shards[1:5], fulls)
    torch.cuda.synchronize()
    for got, ref in zip(fulls, want):
        assert to_np(got).tobytes() == ref.tobytes()
    run.close()


@pytest.mark.parametrize("shapes", [[(256, 64), (64, 8), (512, 16), (1024, 1)],   # bulk-copy form
                                    [(256, 64), (10, 1), (4097, 33)]])           # falls back
def test_group_gather_lean_mode(shapes):
    """With the lean (bulk-copy) gather mode a group gather whose rows are all
    16-byte aligned multiples of 16 bytes runs on the bulk-copy engine, any
    other on the SM kernel; either way the same bytes, and no wait runs out."""
    import zero_sharded_optimizer_step_gb300 as z
    from workloads.runner import Runner, TORCH_DTYPE
    w = W.dim0(shapes, 4, rank=0, steps=1)
    run = Runner(w)
    before = z.zero_gather_timeouts()
    z.zero3_begin_step(run.ctx)
    dt = TORCH_DTYPE[w.param_dtype]
    n = len(shapes)
    outs = {}
    for mode in (z.ZERO_GATHER_FAST, z.ZERO_GATHER_LEAN):
        z.zero_set_gather_mode(run.ctx, mode)
        fulls = [torch.zeros(w.unit_shard(u) * w.world, dtype=dt, device="cuda:0")
                 for u in range(n)]
        z.zero3_gather_group(run.ctx, 0, run.shards[:n], fulls)
        torch.cuda.synchronize()
        outs[mode] = [to_np(f) for f in fulls]
    for a, b in zip(outs[z.ZERO_GATHER_FAST], outs[z.ZERO_GATHER_LEAN]):
        assert a.tobytes() == b.tobytes()
    for u in range(n):                       # the shards themselves, in rank order
        S = w.unit_shard(u)
        for k in range(w.world):
            assert outs[z.ZERO_GATHER_LEAN][u][k * S:(k + 1) * S].tobytes() == \
                to_np(run.shards[u][k]).tobytes()
    assert z.zero_gather_timeouts() == before
    run.close()


@pytest.mark.parametrize("rank,scaled", [(-1, False), (1, False), (-1, True), (2, True)])
def test_group_step_parity(rank, scaled):
    """Runs of units gathered and stepped (or reduced, then one apply) in one
    launch per group, each rank's grads of a group end to end: bit-identical
    to the oracle, with a skipped step when loss-scaled."""
    shapes = [(256, 64), (512, 33), (128, 7), (64, 1), (1024, 3), (8, 5)]
    w = W.dim0(shapes, 4, rank=rank, steps=3, loss_scale=2.0 ** 8 if scaled else 0.0,
               inject=(2, 1) if scaled else None).replace(groups=[2, 3, 1])
    run, ref = run_both(w)
    if scaled and rank < 0:
        assert ref.skips == [False, True, False]
    compare_runner(run, ref, what="groups")
    run.close()


@pytest.mark.parametrize("rank,shadow", [(-1, False), (1, True)])
def test_group_step_adamw_fp16(rank, shadow):
    """Groups with AdamW, fp16 grads and params, loss-scaled (two passes, or
    one pass over two state sets) with a skipped step: the oracle's result
    bit for bit."""
    shapes = [(256, 64), (512, 33), (128, 7), (64, 1)]
    w = W.dim0(shapes, 4, rank=rank, steps=3, loss_scale=2.0 ** 8, inject=(2, 1),
               weight_decay=0.05).replace(groups=[2, 2], grad_dtype=W.F16, param_dtype=W.F16)
    run, ref = run_both(w, shadow=shadow)
    compare_runner(run, ref, what="groups adamw fp16")
    run.close()


@pytest.mark.parametrize("rank", [-1, 2])
def test_group_with_an_empty_unit(rank):
    """A group holding a unit of zero parameters (and units whose shards are
    not multiples of 16 bytes): gathers, steps and the skip as the oracle
    has them."""
    units = [1000, 0, 2000, 44]
    w = W.Workload("gempty", sum(units), 4, 3, W.F16, W.F16, rank=rank, units=units, steps=3,
                   loss_scale=2.0 ** 8, inject=(2, 1)).replace(groups=[3, 1])
    run, ref = run_both(w, shadow=True)
    compare_runner(run, ref, what="group with an empty unit")
    run.close()


def test_group_call_errors():
    import zero_sharded_optimizer_step_gb300 as z
    from workloads.runner import Runner
    shapes = [(256, 64), (10, 1), (64, 7)]          # (10, 1) leaves padding on rank 3
    w = W.dim0(shapes, 4, rank=3, steps=1)
    run = Runner(w)
    z.zero3_begin_step(run.ctx)
    g = [torch.zeros(w.unit_shard(0) + w.unit_shard(1), dtype=torch.bfloat16, device="cuda:0")
         for _ in range(4)]
    with pytest.raises(z.ZeroError) as ei:          # a padded unit in the group
        z.zero3_step_group(run.ctx, 0, 2, g, 1e-3, 0.9, 0.999, 1e-8, 1)
    assert ei.value.code == z.ZERO_EINVAL and "padding" in str(ei.value)
    with pytest.raises(z.ZeroError):                # past the last unit
        z.zero3_step_group(run.ctx, 2, 2, g, 1e-3, 0.9, 0.999, 1e-8, 1)
    with pytest.raises(z.ZeroError):                # wrong number of grad buffers
        z.zero3_step_group(run.ctx, 0, 1, g[:3], 1e-3, 0.9, 0.999, 1e-8, 1)
    with pytest.raises(z.ZeroError):                # shards for the wrong number of units
        z.zero3_gather_group(run.ctx, 0, run.shards[0:2], [run.unit_full])
    z.zero3_step_group(run.ctx, 2, 1, [b[:w.unit_shard(2)] for b in g], 1e-3, 0.9, 0.999,
                       1e-8, 1)                     # a group without padding is fine
    run.close()
    big = W.dim0([(64, 1)] * 130, 4, rank=0, steps=1)   # 130 units x 4 ranks > 512 shards
    run = Runner(big)
    z.zero3_begin_step(run.ctx)
    fulls = [run.unit_full[:64] for _ in range(130)]
    with pytest.raises(z.ZeroError) as ei:
        z.zero3_gather_group(run.ctx, 0, run.shards, fulls)
    assert "512" in str(ei.value)
    run.close()


# ------------------------------- stage 3 in one pass over two state sets

@pytest.mark.parametrize("rank,scaled,layout", [(-1, True, "units"), (1, True, "units"),
                                                (-1, False, "units"), (2, True, "dim0"),
                                                (-1, True, "groups"), (3, True, "hyper")])
def test_stage3_one_pass_two_state_sets(rank, scaled, layout):
    """Loss-scaled ZeRO-3 with a second state set: every unit steps in one
    pass into the other set and zero3_end_step applies the verdict once --
    bit-identical to the oracle (which defers Adam), the +inf step skipped by
    every unit, params recast from the kept set."""
    kw = dict(steps=4, loss_scale=2.0 ** 9 if scaled else 0.0, inject=(2, 1) if scaled else None)
    if layout == "dim0":
        w = W.dim0([(256, 64), (10, 1), (4097, 33), (3, 11)], 4, rank=rank, **kw)
    elif layout == "groups":
        w = W.Workload("s3g", 300_000 + 80_000 + 123_456, 8, 3, W.F16, W.F16, rank=rank,
                       units=[300_000, 80_000, 123_456], groups=[2, 1], **kw)
    else:
        units = [100_003, 7, 250_000, 33_333]
        w = W.Workload("s3s", sum(units), 4, 3, W.F16, W.F16, rank=rank, units=units, **kw)
    run, ref = run_both(w, shadow=True, hyper=layout == "hyper")
    if scaled and rank < 0:
        assert ref.skips == [False, True, False, False]
    compare_runner(run, ref, what="stage3 one pass")
    run.close()


def test_grouped_prefetch_schedule_matches_serial_and_oracle():
    """FSDP2's per-parameter units in layer groups, each group's gather
    prefetched on the background stream (the lean bulk-copy form: every
    shard 16-byte aligned) while the previous group computes: the same
    results as the serial schedule and the oracle."""
    from workloads.runner import Runner
    from workloads.zero3_schedule import Zero3Schedule
    shapes = [(256, 64), (512, 16), (64, 8), (1024, 8), (128, 32)]
    w = W.dim0(shapes, 4, rank=1, steps=3).replace(groups=[2, 2, 1])
    runs = {}
    for mode, bg in (("serial", False), ("overlap", False), ("overlap", True)):
        run = Runner(w)
        sch = Zero3Schedule(run, 2000, 4000, 64, mode, overlap_steps=bg)
        for it in range(1, 4):
            run.fill_grads(it)
            sch.launch_step()
        torch.cuda.synchronize()
        runs[(mode, bg)] = run
    ref = refs.OracleRun(w)
    for it in range(1, 4):
        ref.step(it)
    for key in [("overlap", False), ("overlap", True)]:
        assert torch.equal(runs[("serial", False)].master, runs[key].master)
        assert torch.equal(runs[("serial", False)].params, runs[key].params)
        runs[key].skips = ref.skips
        compare_runner(runs[key], ref, what="grouped prefetch %s" % (key,))
    for run in runs.values():
        run.close()


def test_stage3_one_pass_prefetched_schedule():
    """The prefetch schedule with two state sets: the same results as the
    serial one and the oracle, with a skipped step."""
    from workloads.runner import Runner
    from workloads.zero3_schedule import Zero3Schedule
    units = [200_003, 150_000, 99_999, 250_000]
    w = W.Workload("s3p", sum(units), 4, 3, W.BF16, W.BF16, rank=-1, units=units, steps=4,
                   loss_scale=2.0 ** 10, inject=(2, 1))
    runs = {}
    for mode, bg in (("serial", False), ("overlap", False), ("overlap", True)):
        run = Runner(w, shadow=True)
        sch = Zero3Schedule(run, 2000, 4000, 64, mode, overlap_steps=bg)
        for it in range(1, 5):
            run.fill_grads(it)
            sch.launch_step()
            run.finish_step()
        torch.cuda.synchronize()
        runs[(mode, bg)] = run
    ref = refs.OracleRun(w)
    for it in range(1, 5):
        ref.step(it)
    for run in runs.values():
        assert run.skips == ref.skips == [False, True, False, False]
        compare_runner(run, ref, what="stage3 one pass prefetch")
        run.close()


def test_stage3_two_state_sets_protocol():
    import zero_sharded_optimizer_step_gb300 as z
    from workloads.runner import Runner
    units = [1000, 2000]
    w = W.Workload("s3e", 3000, 4, 3, W.BF16, W.BF16, units=units, steps=1,
                   loss_scale=2.0 ** 8)
    run = Runner(w, shadow=True, scratch=True)
    g = run.grads[0]
    with pytest.raises(z.ZeroError):                 # not begun
        z.zero3_step_unit(run.ctx, 0, g, 1e-3, 0.9, 0.999, 1e-8, 1)
    z.zero3_begin_step_scaled(run.ctx, run.scale)
    with pytest.raises(z.ZeroError):                 # the previous step is still open
        z.zero3_begin_step(run.ctx)
    with pytest.raises(z.ZeroError):                 # the two-pass calls are refused
        z.zero3_reduce_unit(run.ctx, 0, g, run.scale)
    with pytest.raises(z.ZeroError):
        z.zero_step_apply(run.ctx, 1e-3, 0.9, 0.999, 1e-8, 1)
    with pytest.raises(z.ZeroError):                 # no unbinding mid-step
        z.zero_bind_shadow(run.ctx, None, None, None, None)
    z.zero3_step_unit(run.ctx, 0, g, 1e-3, 0.9, 0.999, 1e-8, 1)
    z.zero3_step_unit(run.ctx, 1, run.grads[1], 1e-3, 0.9, 0.999, 1e-8, 1)
    z.zero3_end_step(run.ctx)
    with pytest.raises(z.ZeroError):                 # nothing open any more
        z.zero3_end_step(run.ctx)
    torch.cuda.synchronize()
    assert z.zero_current_state(run.ctx) == 1        # the written set is current
    run.close()
    # one state set: a loss-scaled stage-3 step cannot run in one pass
    run = Runner(w)
    z.zero3_begin_step_scaled(run.ctx, run.scale)
    with pytest.raises(z.ZeroError):
        z.zero3_step_unit(run.ctx, 0, run.grads[0], 1e-3, 0.9, 0.999, 1e-8, 1)
    z.zero3_end_step(run.ctx)                        # a no-op with one set
    run.close()


# ------------------------------------------------------- save and resume

@pytest.mark.parametrize("kind", ["shadow", "two_pass_rank", "stage3"])
def test_resume_from_saved_state(kind):
    """Save after two steps (the second skipped), resume in a new context
    from the copies, run two more steps: bit-identical to the run that
    never stopped (the protocol the header states for zero_bind)."""
    from workloads.runner import Runner
    if kind == "stage3":
        units = [200_003, 99, 150_000]
        w = W.Workload("res3", sum(units), 8, 3, W.BF16, W.BF16, units=units, steps=4,
                       loss_scale=2.0 ** 10, inject=(2, 3))
    else:
        w = W.Workload("res", 500_003, 8, 2, W.F16, W.F16, rank=3 if kind == "two_pass_rank" else -1,
                       steps=4, loss_scale=2.0 ** 12, inject=(2, 3))
    shadow = kind == "shadow"
    whole = Runner(w, shadow=shadow)
    for it in range(1, 5):
        whole.step(it)
    first = Runner(w, shadow=shadow)
    for it in (1, 2):
        first.step(it)
    torch.cuda.synchronize()
    saved = [t.clone() for t in first.state()] + [first.params.clone()]
    t, scale, good, skips = first.t, first.scale, first.good, list(first.skips)
    assert skips == [False, True] or kind == "two_pass_rank"
    first.close()
    resumed = Runner(w, shadow=shadow)      # fresh buffers: flag and cur words zero
    for dst, src in zip([resumed.master, resumed.m, resumed.v, resumed.params], saved):
        dst.copy_(src)
    resumed.t, resumed.scale, resumed.good = t, scale, good
    for it in (3, 4):
        resumed.step(it)
    torch.cuda.synchronize()
    for a, b in zip(resumed.state() + (resumed.params,), whole.state() + (whole.params,)):
        assert torch.equal(a.view(torch.uint8) if a.dtype != torch.float32 else a.view(torch.int32),
                           b.view(torch.uint8) if b.dtype != torch.float32 else b.view(torch.int32))
    assert skips + resumed.skips == whole.skips
    assert resumed.t == whole.t and resumed.scale == whole.scale
    for r in (whole, resumed):
        r.close()


# ------------------------------------------- steps captured in a CUDA graph

def _hyper(run):
    import zero_sharded_optimizer_step_gb300 as z
    d = torch.zeros(z.ZERO_HYPER_BYTES, dtype=torch.uint8, device=run.dev)
    h = torch.zeros(z.ZERO_HYPER_BYTES, dtype=torch.uint8, pin_memory=True)
    z.zero_bind_hyper(run.ctx, d)
    return d, h


@pytest.mark.parametrize("direct", [False, True])
def test_zero3_step_replayed_from_a_cuda_graph(direct):
    """A whole ZeRO-3 step (forward gathers, backward gathers + unit steps)
    captured once and replayed: per-step scalars come from the device block
    refreshed by a memcpy node (or copied straight into the context's
    constant slot), so three replays equal three real steps."""
    import zero_sharded_optimizer_step_gb300 as z
    from workloads.runner import Runner
    units = [100_003, 7, 250_000, 33_333]
    w = W.Workload("z3g", sum(units), 4, 3, W.BF16, W.BF16, rank=1, units=units, steps=3)
    run = Runner(w)
    d, h = _hyper(run)
    if direct:
        z.zero_bind_hyper(run.ctx, z.zero_hyper_slot(run.ctx))
    ref = refs.OracleRun(w)
    U = len(units)

    def body():
        if direct:
            z.zero_load_hyper(run.ctx, h)
        else:
            d.copy_(h, non_blocking=True)
        z.zero3_begin_step(run.ctx)
        for u in range(U):
            z.zero3_gather_unit(run.ctx, u, run.shards[u], run.unit_full, None)
        for u in reversed(range(U)):
            z.zero3_gather_unit(run.ctx, u, run.shards[u], run.unit_full, None)
            z.zero3_step_unit(run.ctx, u, run.grads[u], 0.0, 0.0, 0.0, 0.0, 1, None)

    graph = torch.cuda.CUDAGraph()
    for it in range(1, 4):
        run.fill_grads(it)
        torch.cuda.synchronize()
        z.zero_prepare_step(run.ctx, h, w.lr, w.beta1, w.beta2, w.eps, it)
        if it == 1:                   # the first step runs eagerly, then is captured
            body()
            torch.cuda.synchronize()
            ref.step(it)
            # capture (the capture itself does not run the kernels)
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                with torch.cuda.graph(graph, stream=s):
                    body()
            continue
        graph.replay()
        torch.cuda.synchronize()
        ref.step(it)
    run.t = 3
    run.skips = ref.skips
    compare_runner(run, ref, what="graph z3")
    run.close()


def test_loss_scaled_single_pass_replayed_with_a_skip():
    """The loss-scaled single pass over two state sets in a graph: the +inf
    at iteration 2 is seen by the replayed kernels (they take the step id
    from the block), the step is skipped, the scale halves, later replays
    apply -- bit-identical to the oracle."""
    import zero_sharded_optimizer_step_gb300 as z
    from workloads.runner import Runner
    w = W.Workload("g2", 1_000_003, 8, 2, W.F16, W.F16, steps=4, loss_scale=2.0 ** 12,
                   inject=(2, 3))
    run = Runner(w, shadow=True)
    d, h = _hyper(run)
    ref = refs.OracleRun(w)

    def body():
        d.copy_(h, non_blocking=True)
        z.zero_step(run.ctx, run.grads[0], 0.0, 0.0, 0.0, 0.0, 1, loss_scale=1.0, stream=None)

    graph = torch.cuda.CUDAGraph()
    t = 0
    for it in range(1, 5):
        run.fill_grads(it)
        torch.cuda.synchronize()
        z.zero_prepare_step(run.ctx, h, w.lr, w.beta1, w.beta2, w.eps, t + 1, run.scale)
        if it == 1:
            body()
            torch.cuda.synchronize()
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                with torch.cuda.graph(graph, stream=s):
                    body()
        else:
            graph.replay()
        torch.cuda.synchronize()
        nonfinite, skipped = z.zero_step_status(run.ctx)
        run.skips.append(skipped)
        if not skipped:
            t += 1
        run.scale, run.good = z.zero_scale_update(run.scale, skipped, run.good, 2000)
        ref.step(it)
    assert run.skips == ref.skips == [False, True, False, False]
    compare_runner(run, ref, what="graph shadow")
    run.close()


HYPER_CASES = [(dict(gdt=g, pdt=p), {}) for g, p in
               [(W.BF16, W.BF16), (W.F16, W.F16), (W.F32, W.F32), (W.BF16, W.F32),
                (W.F32, W.BF16), (W.F16, W.BF16), (W.BF16, W.F16), (W.F32, W.F16),
                (W.F16, W.F32)]]
HYPER_CASES += [
    (dict(gdt=W.F16, pdt=W.F16, loss_scale=2.0 ** 10, inject=(2, 3)), {}),            # two passes
    (dict(gdt=W.F16, pdt=W.F16, loss_scale=2.0 ** 10, inject=(2, 3)), {"shadow": True}),
    (dict(gdt=W.BF16, pdt=W.BF16, weight_decay=0.1), {"shadow": True}),               # AdamW
    (dict(gdt=W.F16, pdt=W.F32, rank=5, world=16), {}),
    (dict(gdt=W.BF16, pdt=W.BF16, bucket=100_000, loss_scale=2.0 ** 8, inject=(2, 1)),
     {"shadow": True}),
    (dict(gdt=W.BF16, pdt=W.BF16, bucket=100_000, loss_scale=2.0 ** 8, inject=(2, 1)), {}),
    (dict(gdt=W.BF16, pdt=W.BF16, units=[300_001, 77, 123_456], rank=1), {}),
    (dict(gdt=W.BF16, pdt=W.BF16, units=[300_001, 77, 123_456], loss_scale=2.0 ** 8,
          inject=(2, 2)), {}),
    # groups of units (sizes divisible by the 8 ranks: no padding)
    (dict(gdt=W.BF16, pdt=W.BF16, units=[300_000, 80_000, 123_456], groups=[2, 1]), {}),
    (dict(gdt=W.F16, pdt=W.F16, units=[300_000, 80_000, 123_456], groups=[1, 2],
          loss_scale=2.0 ** 8, inject=(2, 2)), {}),
]


@pytest.mark.parametrize("spec,kw", HYPER_CASES)
def test_device_scalar_block_parity(spec, kw):
    """The kernels compiled to read the step's scalars from a device block
    (the form a CUDA graph replays) over the dtype matrix and every path --
    fused, two passes, two state sets, AdamW, one rank's view, buckets,
    ZeRO-3 units, with and without a skipped step -- run eagerly with the
    block refreshed before each step and junk hyperparameters in the calls:
    bit-identical to the oracle."""
    spec = dict(spec)
    numel = sum(spec["units"]) if "units" in spec else 1_000_003
    w = W.Workload("hyper", numel, spec.pop("world", 8), 3 if "units" in spec else 2,
                   spec.pop("gdt"), spec.pop("pdt"), steps=3, lr=1e-3, **spec)
    run, ref = run_both(w, hyper=True, **kw)
    if w.inject:
        assert True in ref.skips
    compare_runner(run, ref, what="hyper " + str((spec, kw)))
    run.close()


def test_device_scalar_block_unaligned_grads():
    """Grads 2 bytes off a 16-byte boundary take the per-element path of the
    device-block kernels; same result as the oracle."""
    import zero_sharded_optimizer_step_gb300 as z
    from workloads.runner import Runner
    w = W.Workload("hyper-mis", 200_003, 4, 2, W.BF16, W.BF16, steps=2, lr=1e-3)
    run = Runner(w, hyper=True)
    ref = refs.OracleRun(w)
    n = run.grads[0][0].numel()
    for it in (1, 2):
        run.fill_grads(it)
        off = [torch.empty(n + 8, dtype=torch.bfloat16, device=run.dev)[1:1 + n]
               for _ in run.grads[0]]
        for a, b in zip(off, run.grads[0]):
            a.copy_(b)
        run.launch_step(grads_override=off)
        run.finish_step()
        ref.step(it)
    compare_runner(run, ref, what="hyper unaligned")
    z.zero_bind_hyper(run.ctx, None)
    run.close()


def test_constant_slots_are_limited_and_freed():
    """Eight contexts per device may hold a scalar block at once; a ninth is
    refused until one is unbound or destroyed; the device advance refuses a
    block that is the constant slot itself."""
    import zero_sharded_optimizer_step_gb300 as z
    dev = torch.device("cuda:0")
    ctxs, blocks = [], []
    for k in range(9):
        c = z.zero_init(64, 2, 2, z.ZERO_F32, z.ZERO_F32, -1)
        P = z.zero_ctx_state_elems(c)
        bufs = [torch.zeros(P, device=dev) for _ in range(4)]
        flag = torch.zeros(1, dtype=torch.int64, device=dev)
        z.zero_bind(c, *bufs[:3], bufs[3], None, flag)
        ctxs.append((c, bufs, flag))
        blocks.append(torch.zeros(z.ZERO_HYPER_BYTES, dtype=torch.uint8, device=dev))
    for k in range(8):
        z.zero_bind_hyper(ctxs[k][0], blocks[k])
    with pytest.raises(z.ZeroError) as ei:
        z.zero_bind_hyper(ctxs[8][0], blocks[8])
    assert ei.value.code == z.ZERO_ESTATE
    z.zero_bind_hyper(ctxs[3][0], None)              # unbinding frees a slot
    z.zero_bind_hyper(ctxs[8][0], blocks[8])
    with pytest.raises(z.ZeroError):
        z.zero_bind_hyper(ctxs[3][0], blocks[3])
    ctxs[0][0].close()                               # so does destroying a context
    z.zero_bind_hyper(ctxs[3][0], z.zero_hyper_slot(ctxs[3][0]))
    with pytest.raises(z.ZeroError):                 # the advance rewrites its block
        st = torch.zeros(4, dtype=torch.int64, device=dev)
        tab = torch.zeros(8, device=dev)
        z.zero_bind_advance(ctxs[3][0], tab, 4, st)
        h = torch.zeros(z.ZERO_HYPER_BYTES, dtype=torch.uint8, pin_memory=True)
        z.zero_prepare_step(ctxs[3][0], h, 1e-3, 0.9, 0.999, 1e-8, 1)
        z.zero_advance_step(ctxs[3][0])
    for c, _, _ in ctxs[1:]:
        c.close()


def test_prepared_step_protocol():
    import zero_sharded_optimizer_step_gb300 as z
    from workloads.runner import Runner
    w = W.Workload("gp", 1000, 4, 2, W.BF16, W.BF16, steps=1)
    run = Runner(w)
    d, h = _hyper(run)
    with pytest.raises(z.ZeroError):          # not prepared yet
        z.zero_step(run.ctx, run.grads[0], 1e-3, 0.9, 0.999, 1e-8, 1)
    z.zero_prepare_step(run.ctx, h, 1e-3, 0.9, 0.999, 1e-8, 1)
    with pytest.raises(z.ZeroError):          # loss scaling differs from the prepared step
        z.zero_step(run.ctx, run.grads[0], 1e-3, 0.9, 0.999, 1e-8, 1, loss_scale=8.0)
    z.zero_bind_hyper(run.ctx, None)
    run.close()


# ----------------------------------------- scalars advanced on the device

def _advance_setup(run, w, T, growth_interval):
    import zero_sharded_optimizer_step_gb300 as z
    d = torch.zeros(z.ZERO_HYPER_BYTES, dtype=torch.uint8, device=run.dev)
    h = torch.zeros(z.ZERO_HYPER_BYTES, dtype=torch.uint8, pin_memory=True)
    z.zero_bind_hyper(run.ctx, d)
    tab = np.zeros(2 * T, np.float32)
    z.zero_fill_advance_table(tab.ctypes.data, T, w.beta1, w.beta2)
    dtab = torch.from_numpy(tab).to(run.dev)
    hs = np.zeros(4, np.int64)
    z.zero_advance_state(hs.ctypes.data, 1, run.scale, growth_interval)
    ds = torch.from_numpy(hs).to(run.dev)
    z.zero_bind_advance(run.ctx, dtab, T, ds)
    z.zero_prepare_step(run.ctx, h, w.lr, w.beta1, w.beta2, w.eps, 1, run.scale)
    d.copy_(h)
    torch.cuda.synchronize()
    return d, h, dtab, ds


def _state(ds):
    raw = ds.cpu().numpy()
    return (int(raw[0]), float(np.frombuffer(raw[1].tobytes()[:4], np.float32)[0]),
            int(np.frombuffer(raw[1].tobytes()[4:], np.int32)[0]), int(raw[2]))


@pytest.mark.parametrize("graph", [False, True])
def test_device_advance_matches_the_host_policy(graph):
    """Loss-scaled steps whose t, loss scale and bias corrections advance on
    the device (no verdict read back): a skipped step, two growths
    (growth_interval 2), bit-identical to the oracle stepping with the host
    policy; as eager launches and as one CUDA graph of [step, advance]
    replayed step after step."""
    import zero_sharded_optimizer_step_gb300 as z
    from workloads.runner import Runner
    w = W.Workload("adv", 1_000_003, 8, 2, W.F16, W.F16, steps=7, loss_scale=2.0 ** 12,
                   inject=(3, 2), growth_interval=2)
    run = Runner(w, shadow=True)
    d, h, dtab, ds = _advance_setup(run, w, 32, 2)
    ref = refs.OracleRun(w)
    s = torch.cuda.Stream()

    def body():
        z.zero_step(run.ctx, run.grads[0], 0.0, 0.0, 0.0, 0.0, 1, loss_scale=1.0, stream=s)
        z.zero_advance_step(run.ctx, s)

    g = torch.cuda.CUDAGraph() if graph else None
    for it in range(1, 8):
        run.scale = ref.scale                 # the grads are drawn at the scale in force
        run.fill_grads(it)
        torch.cuda.synchronize()
        if graph and it == 1:
            with torch.cuda.stream(s):
                body()
            torch.cuda.synchronize()
            with torch.cuda.stream(s):
                with torch.cuda.graph(g, stream=s):
                    body()
        elif graph:
            with torch.cuda.stream(s):
                g.replay()
        else:
            with torch.cuda.stream(s):
                body()
        torch.cuda.synchronize()
        ref.step(it)
        t, scale, status, good = _state(ds)
        assert (t, scale, status) == (ref.t + 1, ref.scale, 0), (it, t, scale, ref.t, ref.scale)
        assert good == ref.good
    assert ref.skips == [False, False, True, False, False, False, False]
    compare_runner(run, ref, what="device advance" + (" graph" if graph else ""))
    run.close()


def test_device_advance_stops_when_the_table_runs_out():
    """With bias corrections for 3 steps only, the advance after step 3 sets
    the status and leaves the block as it was; nothing faults."""
    import zero_sharded_optimizer_step_gb300 as z
    from workloads.runner import Runner
    w = W.Workload("advT", 10_001, 4, 2, W.BF16, W.BF16, steps=4)
    run = Runner(w)
    d, h, dtab, ds = _advance_setup(run, w, 3, 0)
    for it in (1, 2, 3):
        run.fill_grads(it)
        z.zero_step(run.ctx, run.grads[0], 0.0, 0.0, 0.0, 0.0, 1)
        before = d.cpu().clone()
        z.zero_advance_step(run.ctx)
        torch.cuda.synchronize()
        t, scale, status, good = _state(ds)
        if it < 3:
            assert (t, status) == (it + 1, 0)
        else:
            assert status == 1 and t == 3
            assert torch.equal(d.cpu(), before)
    run.close()


def _direct_step_case(grads_h, gdt, pdt, scale, x0, steps, shadow, hp=(1e-3, 0.9, 0.999, 1e-8),
                      t0=0):
    """Steps the same host grads through zero_step (all ranks) and through
    the oracle; returns the GPU verdicts and asserts bit-identity."""
    import zero_sharded_optimizer_step_gb300 as z
    dev = torch.device("cuda:0")
    world, numel = len(grads_h), grads_h[0].size
    c = z.zero_init(numel, world, 2, gdt, pdt, -1)
    P = z.zero_ctx_state_elems(c)
    xh = np.zeros(P, np.float32)
    xh[:numel] = x0
    mh, vh = np.zeros(P, np.float32), np.zeros(P, np.float32)
    ph = np.zeros(P, STORAGE[pdt])
    ph[:] = oracle.cast(xh, pdt)
    tdt = {W.F32: torch.float32, W.BF16: torch.bfloat16, W.F16: torch.float16}
    master = torch.from_numpy(xh.copy()).to(dev)
    m, v = torch.zeros(P, device=dev), torch.zeros(P, device=dev)
    params = torch.from_numpy(ph.copy().view(np.int16) if pdt != W.F32 else ph.copy()).to(dev)
    if pdt != W.F32:
        params = params.view(tdt[pdt])
    flag = torch.zeros(1, dtype=torch.int64, device=dev)
    scratch = None if shadow else torch.zeros(P, device=dev)
    z.zero_bind(c, master, m, v, params, scratch, flag)
    if shadow:
        sh = (master.clone(), torch.zeros(P, device=dev), torch.zeros(P, device=dev),
              torch.zeros(1, dtype=torch.int64, device=dev))
        z.zero_bind_shadow(c, *sh)
    gd = []
    for g in grads_h:
        t = torch.from_numpy(g.view(np.int16) if gdt != W.F32 else g).to(dev)
        gd.append(t.view(tdt[gdt]) if gdt != W.F32 else t)
    verdicts, t = [], t0
    for _ in range(steps):
        z.zero_step(c, gd, *hp, t + 1, scale)
        _, skipped = z.zero_step_status(c)
        o_skip, _ = oracle.zero_step(grads_h, gdt, numel, xh, mh, vh, ph, pdt, *hp, t + 1,
                                     loss_scale=scale)
        assert skipped == o_skip
        verdicts.append(skipped)
        t += 0 if skipped else 1
    cur = z.zero_current_state(c) if shadow else 0
    cx, cm, cv = (sh[:3] if cur == 1 else (master, m, v))
    for name, a, b in [("master", to_np(cx), xh), ("m", to_np(cm), mh), ("v", to_np(cv), vh)]:
        assert_bit_identical(a, b, oracle.F32, name)
    assert_bit_identical(to_np(params), ph, pdt, "params")
    c.close()
    return verdicts


@pytest.mark.parametrize("shadow", [False, True])
def test_loss_scale_edge_values(shadow):
    """(1) A loss scale that is not a power of two (3000): the unscale is a
    true division on both sides.  (2) A scale of 2^-8 (allowed: its inverse
    is normal) with finite sums near 2^120: the sum is finite but the
    unscaled grad overflows, and the step is skipped.  (3) bf16 grads of
    2^127 in every rank: each is finite, their fp32 sum is not, and the step
    is skipped.  Each against the oracle, bit for bit."""
    rng = np.random.default_rng(7)
    n, world = 70_001, 4
    x0 = synth.fill_host(n, synth.F32, synth.key(3, synth.KIND_MASTER), 0.01)

    def draws(scale, dtype):
        return [synth.fill_host(n, dtype, synth.key(3, synth.KIND_GRAD, 1, k), 1e-3 * scale)
                for k in range(world)]

    # (1) non-power-of-two scale, fp16 grads: applied, division path
    g = draws(3000.0, W.F16)
    assert _direct_step_case(g, W.F16, W.F16, 3000.0, x0, 2, shadow) == [False, False]
    # (2) scale 2^-8: one element's sum ~2^121 is finite, /N then *2^8 overflows
    g = [a.copy() for a in draws(1.0, W.F32)]
    e = int(rng.integers(0, n))
    for k in range(world):
        g[k][e] = np.float32(2.0 ** 120)
    assert _direct_step_case(g, W.F32, W.BF16, 2.0 ** -8, x0, 1, shadow) == [True]
    # the same grads at scale 1 are applied (2^122 / 4 is finite)
    assert _direct_step_case(g, W.F32, W.BF16, 1.0, x0, 1, shadow) == [False]
    # (3) bf16 grads 2^127 in every rank at one position: the fp32 sum overflows
    g = [a.copy() for a in draws(2.0 ** 10, W.BF16)]
    big = oracle.cast(np.array([2.0 ** 127], np.float32), W.BF16)[0]
    for k in range(world):
        g[k][e] = big
    assert _direct_step_case(g, W.BF16, W.BF16, 2.0 ** 10, x0, 1, shadow) == [True]


@pytest.mark.parametrize("pdt", [W.F32, W.BF16, W.F16])
def test_subnormals_are_kept(pdt):
    """No flush to zero anywhere: fp32 grads around 1e-20 make g*g and v
    subnormal (about 1e-43), and masters around 1e-39 are subnormal fp32
    (and bf16) values that the cast must round, not flush.  Bit-identical
    to the oracle, which runs on the host FPU with subnormals."""
    n, world = 50_001, 3
    x0 = synth.fill_host(n, synth.F32, synth.key(5, synth.KIND_MASTER), 0.01)
    tiny = synth.fill_host(n, synth.F32, synth.key(5, synth.KIND_MASTER, 1), 1e-39)
    x0[::3] = tiny[::3]
    g = [synth.fill_host(n, W.F32, synth.key(5, synth.KIND_GRAD, 1, k), 1e-20)
         for k in range(world)]
    assert (np.abs(x0[::3]) < np.finfo(np.float32).tiny).mean() > 0.9
    sq = g[0].astype(np.float32) * g[0].astype(np.float32)
    assert ((sq != 0) & (np.abs(sq) < np.finfo(np.float32).tiny)).mean() > 0.5
    assert _direct_step_case(g, W.F32, pdt, 0.0, x0, 3, False) == [False] * 3


@pytest.mark.parametrize("hp,t0", [
    ((0.0, 0.9, 0.999, 1e-8), 0),          # lr 0: masters and params unchanged, m and v move
    ((1e-3, 0.0, 0.0, 1e-8), 0),           # no momentum: m = g, v = g*g
    ((1e-3, 0.9, 0.999, 0.0), 0),          # eps 0: the step is lr * mh / sqrt(vh)
    ((1e-2, 0.9, 0.999, 1e-8), 999_997),   # t near 10^6: bias corrections round to 1
    ((1e-3, 0.5, 0.5, 1e-3), 1_100),       # 0.5^t underflows double: corrections exactly 1
])
def test_extreme_valid_hyperparameters(hp, t0):
    """Values at the edges of the ranges Adam is defined on, bit-identical to
    the oracle over three steps (fp32 grads, bf16 params)."""
    n, world = 40_003, 3
    x0 = synth.fill_host(n, synth.F32, synth.key(6, synth.KIND_MASTER), 0.01)
    g = [synth.fill_host(n, W.F32, synth.key(6, synth.KIND_GRAD, 1, k), 1e-3) for k in range(world)]
    assert _direct_step_case(g, W.F32, W.BF16, 0.0, x0, 3, False, hp=hp, t0=t0) == [False] * 3
