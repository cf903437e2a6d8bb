"""The sharded step with libzero.so doing each rank's arithmetic: two
processes, each one data-parallel rank in the one-rank view (LibraryRank)
driven by ShardedStep, their data exchanged by gloo through host memory
(this run has one GPU, so both processes use it; no kernel of one process
waits for the other's).  The result must be bit-identical to the oracle's
all-ranks step: the state of every shard, the full parameter buffer every
rank ends with, and the skip of the step that holds a +inf -- with two
state sets and with the fp32 scratch, loss-scaled and not."""
import os

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from tests.test_multiprocess_gloo import _all_ranks_reference, _free_port

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, numel, inject_at, shadow, out_dir, weight_decay=0.0, bucket=0,
          stage=2):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import oracle
    import synth
    import zero_sharded_optimizer_step_gb300 as z
    from zero_sharded_optimizer_step_gb300.sharded import LibraryRank, ShardedStep
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    torch.cuda.set_device(0)
    local = LibraryRank(numel, world, rank, z.ZERO_F16, z.ZERO_F16, "cuda:0", shadow=shadow,
                        weight_decay=weight_decay, stage=stage)
    S = local.shard
    lo = rank * S
    nv = max(0, min(S, numel - lo))
    x0 = np.zeros(S, np.float32)
    x0[:nv] = synth.fill_host(nv, synth.F32, synth.key(0, synth.KIND_MASTER), 0.01, index0=lo)
    local.set_master(torch.from_numpy(x0).cuda())
    step = ShardedStep(local)
    P = S * world
    scale, good, t, skips = 2.0 ** 12, 0, 0, []
    for it in (1, 2, 3):
        g = np.zeros(P, np.uint16)
        g[:numel] = synth.fill_host(numel, synth.F16, synth.key(0, synth.KIND_GRAD, it, rank),
                                    1e-3 * scale)
        if inject_at and it == inject_at[0] and rank == inject_at[1]:
            g[inject_at[2]] = 0x7C00                          # +inf in fp16
        dg = torch.from_numpy(g.view(np.int16)).cuda().view(torch.float16)
        if bucket:
            # bucket by bucket from one reused device buffer
            buf = torch.zeros(bucket, dtype=torch.float16, device="cuda:0")
            step.begin(scale)
            for off in range(0, P, bucket):
                n = min(bucket, P - off)
                buf[:n].copy_(dg[off:off + n])
                step.bucket(off, buf[:n], 1e-3, 0.9, 0.999, 1e-8, t + 1)
            _, skipped = step.end(1e-3, 0.9, 0.999, 1e-8, t + 1)
        else:
            _, skipped = step.step(dg, 1e-3, 0.9, 0.999, 1e-8, t + 1, loss_scale=scale)
        skips.append(skipped)
        if not skipped:
            t += 1
        scale, good = oracle.scale_update(scale, skipped, good, 2000)
    torch.cuda.synchronize()
    x, m, v = (a.cpu().numpy() for a in local.state())
    full = local.params.cpu().view(torch.int16).numpy().view(np.uint16)
    extra = {}
    if stage == 1:
        extra["avg"] = local.grad_avg.cpu().view(torch.int16).numpy().view(np.uint16)
    np.savez(os.path.join(out_dir, "rank%d.npz" % rank), x=x, m=m, v=v, full=full,
             skips=np.array(skips), **extra)
    local.close()
    dist.destroy_process_group()


@pytest.mark.parametrize("numel,inject_at,shadow,bucket", [
    (300_007, None, True, 0),
    (300_007, (2, 1, 299_999), True, 0),      # rank 1's +inf in rank 1's shard
    (300_007, (2, 0, 200_001), False, 0),     # rank 0's +inf in rank 1's shard
    (300_007, (2, 0, 200_001), True, 70_001),  # buckets, one across the shard boundary
    (300_007, (2, 1, 299_999), False, 70_001),
])
def test_sharded_step_through_the_library(tmp_path, numel, inject_at, shadow, bucket):
    world = 2
    port = _free_port()
    mp.start_processes(_rank, args=(world, port, numel, inject_at, shadow, str(tmp_path), 0.0,
                                    bucket), nprocs=world, join=True, start_method="spawn")
    import oracle
    x, m, v, full, skips = _all_ranks_reference(numel, world, inject_at)
    assert skips == [bool(inject_at) and it == inject_at[0] for it in (1, 2, 3)]
    S = oracle.shard_size(numel, world)
    for r in range(world):
        d = np.load(os.path.join(tmp_path, "rank%d.npz" % r))
        assert list(d["skips"]) == skips, r
        sl = slice(r * S, (r + 1) * S)
        assert d["x"].tobytes() == x[sl].tobytes()
        assert d["m"].tobytes() == m[sl].tobytes()
        assert d["v"].tobytes() == v[sl].tobytes()
        assert d["full"].tobytes() == full.tobytes()


def _ranks(proc, nprocs, port, numel, world, inject_at, shadow, out_dir, stage=2):
    """Process `proc` of `nprocs` holding world // nprocs consecutive ranks
    in the library's view of several ranks (LibraryRank(n_ranks=k)), driven
    by RanksStep."""
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import oracle
    import synth
    import zero_sharded_optimizer_step_gb300 as z
    from zero_sharded_optimizer_step_gb300.sharded import LibraryRank, RanksStep
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=proc, world_size=nprocs)
    torch.cuda.set_device(0)
    k = world // nprocs
    local = LibraryRank(numel, world, proc * k, z.ZERO_F16, z.ZERO_F16, "cuda:0",
                        shadow=shadow, stage=stage, n_ranks=k)
    S = local.shard
    P = S * world
    lo = proc * k * S
    nv = max(0, min(k * S, numel - lo))
    x0 = np.zeros(k * S, np.float32)
    x0[:nv] = synth.fill_host(nv, synth.F32, synth.key(0, synth.KIND_MASTER), 0.01, index0=lo)
    local.set_master(torch.from_numpy(x0).cuda())
    step = RanksStep(local)
    scale, good, t, skips = 2.0 ** 12, 0, 0, []
    for it in (1, 2, 3):
        dgs = []
        for c in range(k):
            g = np.zeros(P, np.uint16)
            g[:numel] = synth.fill_host(numel, synth.F16,
                                        synth.key(0, synth.KIND_GRAD, it, proc * k + c),
                                        1e-3 * scale)
            if inject_at and it == inject_at[0] and proc * k + c == inject_at[1]:
                g[inject_at[2]] = 0x7C00
            dgs.append(torch.from_numpy(g.view(np.int16)).cuda().view(torch.float16))
        _, skipped = step.step(dgs, 1e-3, 0.9, 0.999, 1e-8, t + 1, loss_scale=scale)
        skips.append(skipped)
        if not skipped:
            t += 1
        scale, good = oracle.scale_update(scale, skipped, good, 2000)
    torch.cuda.synchronize()
    full = local.params.cpu().view(torch.int16).numpy().view(np.uint16)
    x, m, v = (a.cpu().numpy() for a in local.state())
    extra = {}
    if stage == 1:
        extra["avg"] = local.grad_avg.cpu().view(torch.int16).numpy().view(np.uint16)
    for c in range(k):
        sl = slice(c * S, (c + 1) * S)
        np.savez(os.path.join(out_dir, "rank%d.npz" % (proc * k + c)), x=x[sl], m=m[sl],
                 v=v[sl], full=full, skips=np.array(skips), **extra)
    local.close()
    dist.destroy_process_group()


@pytest.mark.parametrize("nprocs,world,numel,inject_at,shadow,stage", [
    (1, 4, 300_007, (2, 3, 17), True, 2),        # every rank in one view, no collective
    (1, 4, 300_007, (2, 1, 299_999), False, 2),  # the fp32 scratch
    (1, 4, 300_013, (2, 2, 75_011), True, 2),    # S = 4 mod 8
    (2, 4, 300_007, (2, 3, 17), True, 2),        # two ranks in each of two processes
    (2, 4, 300_013, None, False, 2),
    (2, 6, 300_001, (2, 5, 1), False, 2),
    (2, 4, 300_013, None, True, 1),              # stage 1: the averaged grads gathered too
])
def test_ranks_per_process_through_the_library(tmp_path, nprocs, world, numel, inject_at,
                                               shadow, stage):
    """W ranks over N processes, each process one library view of its W/N
    ranks (RanksStep): with N = 1 the view holds every rank and the step is
    one pass with no collective; with N = 2 each rank's pieces are exchanged
    between the processes.  The state of every rank, the full parameter
    buffer (and, stage 1, the averaged grads) and the skips bit-identical to
    the oracle's all-ranks step."""
    port = _free_port()
    mp.start_processes(_ranks, args=(nprocs, port, numel, world, inject_at, shadow,
                                     str(tmp_path), stage), nprocs=nprocs, join=True,
                       start_method="spawn")
    import oracle
    import synth
    x, m, v, full, skips = _all_ranks_reference(numel, world, inject_at)
    assert skips == [bool(inject_at) and it == inject_at[0] for it in (1, 2, 3)]
    S = oracle.shard_size(numel, world)
    avg = None
    if stage == 1:
        # no overflow: the scale stays 2^12 and step 3's grads are these
        grads = [synth.fill_host(numel, synth.F16, synth.key(0, synth.KIND_GRAD, 3, k),
                                 1e-3 * 2.0 ** 12) for k in range(world)]
        avg = oracle.cast(oracle.all_reduce_mean(grads, oracle.F16, numel), oracle.F16)
    for r in range(world):
        d = np.load(os.path.join(tmp_path, "rank%d.npz" % r))
        assert list(d["skips"]) == skips, r
        sl = slice(r * S, (r + 1) * S)
        assert d["x"].tobytes() == x[sl].tobytes(), r
        assert d["m"].tobytes() == m[sl].tobytes(), r
        assert d["v"].tobytes() == v[sl].tobytes(), r
        assert d["full"].tobytes() == full.tobytes(), r
        if avg is not None:
            assert d["avg"].tobytes() == avg.tobytes(), r


@pytest.mark.parametrize("extra,updated", [
    (["--numel", "4000037"], 16 * (-(-4000037 // 16))),
    (["--numel", "4000037", "--dp-ranks", "2"], 2 * (-(-4000037 // 2))),
    (["--workload", "zero3_gpt2_small"], None),
])
def test_bench_sharded_mode_runs(extra, updated):
    """bench.py's default mode for --gpus 2 under torchrun: two gloo
    processes on this GPU, a small flat vector over the workload's 16 ranks
    (8 per process) or over 2 (one each), and the 14 ZeRO-3 units of GPT-2
    small over its 8 ranks (4 per process); the line reports strong scaling
    and every step applied."""
    import json
    import subprocess
    import sys

    import workloads as W
    port = _free_port()
    out = subprocess.run(
        [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
         "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--gpus", "2",
         "--dist-backend", "gloo", "--steps", "2", "--warmup", "3", *extra],
        cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2 and d["scaling"] == "strong" and d["value"] > 0
    if updated is None:
        w = W.zero3_gpt2_small()               # its own 8 ranks, 4 per process
        updated = w.world * sum(w.unit_shard(u) for u in range(len(w.units)))
    assert d["config"]["params_updated_per_step"] == updated
    assert "gloo" in d["config"]["parallelism"]
    assert 0.0 <= d["measured"]["collective_share_of_step"] <= 1.0
    assert d["e2e"]["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] > 0
    assert d["e2e"]["d2h_bytes_per_step"] > 0


def _rank3(proc, nprocs, world, port, units, inject_at, shadow, out_dir, prefetch=False):
    """Process `proc` of `nprocs`, holding world // nprocs consecutive ranks
    of a ZeRO-3 step (LibraryRank3, one rank's view or a view of several)."""
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import oracle
    import synth
    import zero_sharded_optimizer_step_gb300 as z
    from zero_sharded_optimizer_step_gb300.sharded import LibraryRank3, ShardedZero3Step
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=proc, world_size=nprocs)
    torch.cuda.set_device(0)
    k = world // nprocs
    first = proc * k
    local = LibraryRank3(units, world, first, z.ZERO_F16, z.ZERO_F16, "cuda:0", shadow=shadow,
                         n_ranks=k)
    for u, (nu, S) in enumerate(zip(units, local.shards)):
        nv = max(0, min(k * S, nu - first * S))
        x = np.zeros(k * S, np.float32)
        x[:nv] = synth.fill_host(nv, synth.F32, synth.key(0, synth.KIND_MASTER, 0, 0, u), 0.01,
                                 index0=first * S)
        local.set_master(u, torch.from_numpy(x).cuda())
    step = ShardedZero3Step(local, prefetch=prefetch)
    scale, good, t, skips, gathered = 2.0 ** 12, 0, 0, [], {}
    for it in (1, 2, 3):
        def forward(u, params):
            gathered[u] = params.cpu().view(torch.int16).numpy().view(np.uint16).copy()

        def backward(u, params):
            gathered[u] = params.cpu().view(torch.int16).numpy().view(np.uint16).copy()
            nu, S = units[u], local.shards[u]
            out = []
            for c in range(k):
                r = first + c
                g = np.zeros(S * world, np.uint16)
                g[:nu] = synth.fill_host(nu, synth.F16, synth.key(0, synth.KIND_GRAD, it, r, u),
                                         1e-3 * scale)
                if inject_at and (it, r, u) == inject_at[:3]:
                    g[inject_at[3]] = 0x7C00              # +inf in fp16
                out.append(torch.from_numpy(g.view(np.int16)).cuda().view(torch.float16))
            return out if k > 1 else out[0]
        _, skipped = step.step(backward, 1e-3, 0.9, 0.999, 1e-8, t + 1, loss_scale=scale,
                               forward=forward)
        skips.append(skipped)
        if not skipped:
            t += 1
        scale, good = oracle.scale_update(scale, skipped, good, 2000)
    torch.cuda.synchronize()
    cx, cm, cv = (a.cpu().numpy() for a in local.state())
    for j in range(k):
        out = {"skips": np.array(skips)}
        for u in range(len(units)):
            S = local.shards[u]
            o = local.offsets[u] + j * S
            out["x%d" % u], out["m%d" % u], out["v%d" % u] = cx[o:o + S], cm[o:o + S], cv[o:o + S]
            lp = local.own_params(u).cpu().view(torch.int16).numpy().view(np.uint16)
            out["lp%d" % u] = lp[j * S:(j + 1) * S]
            out["full%d" % u] = gathered[u]
        np.savez(os.path.join(out_dir, "rank%d.npz" % (first + j)), **out)
    local.close()
    dist.destroy_process_group()


@pytest.mark.parametrize("nprocs,world,inject_at,shadow,prefetch", [
    (2, 2, None, True, False),
    (2, 2, (2, 1, 0, 1400), True, False),    # (iteration, rank, unit, element)
    (2, 2, (2, 0, 2, 4001), False, False),   # rank 0's element in rank 1's shard of unit 2
    (2, 2, (2, 1, 0, 1400), True, True),     # the next unit's gather in flight
    (2, 2, None, False, True),
    (1, 4, (2, 3, 2, 11), True, False),      # every rank in one process: the library gathers
    (1, 4, (2, 1, 0, 1400), False, True),
    (2, 4, (2, 3, 2, 11), True, True),       # two ranks in each of two processes
    (1, 3, (2, 2, 1, 16), True, False),      # padding in every unit
])
def test_sharded_zero3_through_the_library(tmp_path, nprocs, world, inject_at, shadow, prefetch):
    """ZeRO-3 across processes (ShardedZero3Step over LibraryRank3), one rank
    or several per process: per unit an all-gather before forward and
    backward (with one process, the library's placement), the unit's grads
    exchanged after its backward and stepped, every unit's verdict combined
    -- bit-identical to the oracle's all-ranks step of every unit."""
    from tests.test_multiprocess_gloo import _stage3_reference
    units = [3001, 17, 5000]
    port = _free_port()
    mp.start_processes(_rank3, args=(nprocs, world, port, units, inject_at, shadow, str(tmp_path),
                                     prefetch), nprocs=nprocs, join=True, start_method="spawn")
    import oracle
    st, fulls, skips = _stage3_reference(units, world, inject_at)
    assert skips == [bool(inject_at) and it == 2 for it in (1, 2, 3)]
    first = None
    for r in range(world):
        d = np.load(os.path.join(tmp_path, "rank%d.npz" % r))
        assert list(d["skips"]) == skips, r
        for u, nu in enumerate(units):
            S = oracle.shard_size(nu, world)
            sl = slice(r * S, (r + 1) * S)
            for name, a in zip("xmv", st[u]):
                assert d["%s%d" % (name, u)].tobytes() == a[sl].tobytes(), (r, u, name)
            assert d["lp%d" % u].tobytes() == fulls[u][sl].tobytes()
        if first is None:
            first = {u: d["full%d" % u].copy() for u in range(len(units))}
        else:
            for u in range(len(units)):
                assert d["full%d" % u].tobytes() == first[u].tobytes()


def _nccl_one_rank(index, port, out_dir):
    """A process group of one over NCCL: every collective the sharded steps
    make (the byte all-to-all, the int64 MAX all-reduce, the in-place
    all-gather) runs through the NCCL backend on this GPU."""
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import synth
    import zero_sharded_optimizer_step_gb300 as z
    from zero_sharded_optimizer_step_gb300.sharded import (LibraryRank, LibraryRank3,
                                                           ShardedStep, ShardedZero3Step)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", rank=0, world_size=1)
    assert dist.get_backend() == "nccl"
    numel = 100_003
    local = LibraryRank(numel, 1, 0, z.ZERO_BF16, z.ZERO_BF16, "cuda:0", shadow=True)
    x0 = synth.fill_host(numel, synth.F32, synth.key(5, synth.KIND_MASTER), 0.01)
    local.set_master(torch.from_numpy(x0).cuda())
    step = ShardedStep(local)
    g = synth.fill_host(numel, synth.BF16, synth.key(5, synth.KIND_GRAD, 1, 0), 1e-3)
    dg = torch.from_numpy(g.view(np.int16)).cuda().view(torch.bfloat16)
    verdict = step.step(dg, 1e-3, 0.9, 0.999, 1e-8, 1, loss_scale=256.0)
    torch.cuda.synchronize()
    x, m, v = (a.cpu().numpy() for a in local.state())
    p = local.params.cpu().view(torch.int16).numpy().view(np.uint16)
    units = [30_001, 7, 50_000]
    l3 = LibraryRank3(units, 1, 0, z.ZERO_BF16, z.ZERO_BF16, "cuda:0", shadow=False)
    g3 = []
    for u, nu in enumerate(units):
        xu = synth.fill_host(nu, synth.F32, synth.key(5, synth.KIND_MASTER, 0, 0, u), 0.01)
        l3.set_master(u, torch.from_numpy(xu).cuda())
        gu = synth.fill_host(nu, synth.BF16, synth.key(5, synth.KIND_GRAD, 1, 0, u), 1e-3)
        g3.append(torch.from_numpy(gu.view(np.int16)).cuda().view(torch.bfloat16))
    seen = {}

    def backward(u, params):
        seen[u] = params.cpu().view(torch.int16).numpy().view(np.uint16).copy()
        return g3[u]
    # in a group of one the stage-3 step places with the library's gather
    verdict3 = ShardedZero3Step(l3, prefetch=True).step(backward, 1e-3, 0.9, 0.999, 1e-8, 1)
    torch.cuda.synchronize()
    x3, m3, v3 = (a.cpu().numpy() for a in l3.state())
    # the asynchronous all-gather (the prefetch's collective across
    # processes) through NCCL: unit 2's shard into a buffer of its own
    from zero_sharded_optimizer_step_gb300.sharded import gather_params
    agb = torch.zeros_like(l3.own_params(2))
    pending = gather_params(agb, l3.own_params(2), async_op=True)
    pending.wait()
    torch.cuda.synchronize()
    async_ok = torch.equal(agb, l3.own_params(2))
    # the bucketed form (the split-size all-to-all) over NCCL: the same step
    # as above from a fresh rank, in buckets of 30,001
    lb = LibraryRank(numel, 1, 0, z.ZERO_BF16, z.ZERO_BF16, "cuda:0", shadow=True)
    lb.set_master(torch.from_numpy(x0).cuda())
    sb = ShardedStep(lb)
    sb.begin(256.0)
    for off in range(0, numel, 30_001):
        sb.bucket(off, dg[off:off + 30_001], 1e-3, 0.9, 0.999, 1e-8, 1)
    verdict_b = sb.end(1e-3, 0.9, 0.999, 1e-8, 1)
    torch.cuda.synchronize()
    xb = lb.state()[0].cpu().numpy()
    pb = lb.params.cpu().view(torch.int16).numpy().view(np.uint16)
    np.savez(os.path.join(out_dir, "nccl.npz"), x=x, m=m, v=v, p=p, verdict=np.array(verdict),
             xb=xb, pb=pb, verdict_b=np.array(verdict_b),
             x3=x3, p3=l3.params.cpu().view(torch.int16).numpy().view(np.uint16),
             verdict3=np.array(verdict3), async_ok=np.array(async_ok),
             **{"seen%d" % u: s for u, s in seen.items()})
    local.close()
    l3.close()
    lb.close()
    dist.destroy_process_group()


def test_sharded_steps_over_a_one_rank_nccl_group(tmp_path):
    """ShardedStep (whole and bucketed) and ShardedZero3Step (prefetching)
    in a real NCCL group of one rank: the result is the oracle's (one rank:
    the step on the whole vector).  ShardedStep's collectives and the
    asynchronous all-gather run through NCCL; the stage-3 step of a group of
    one places with the library."""
    mp.start_processes(_nccl_one_rank, args=(_free_port(), str(tmp_path)), nprocs=1, join=True,
                       start_method="spawn")
    import oracle
    import synth
    d = np.load(os.path.join(tmp_path, "nccl.npz"))
    numel = 100_003
    x = synth.fill_host(numel, synth.F32, synth.key(5, synth.KIND_MASTER), 0.01)
    m, v = np.zeros(numel, np.float32), np.zeros(numel, np.float32)
    full = np.zeros(numel, np.uint16)
    g = synth.fill_host(numel, synth.BF16, synth.key(5, synth.KIND_GRAD, 1, 0), 1e-3)
    oracle.zero_step([g], oracle.BF16, numel, x, m, v, full, oracle.BF16, 1e-3, 0.9, 0.999, 1e-8,
                     1, loss_scale=256.0)
    assert tuple(d["verdict"]) == (False, False)
    assert d["x"].tobytes() == x.tobytes() and d["m"].tobytes() == m.tobytes()
    assert d["v"].tobytes() == v.tobytes() and d["p"].tobytes() == full.tobytes()
    # the bucketed step: the same result
    assert tuple(d["verdict_b"]) == (False, False)
    assert d["xb"].tobytes() == x.tobytes() and d["pb"].tobytes() == full.tobytes()
    units = [30_001, 7, 50_000]
    xs, ps = [], []
    for u, nu in enumerate(units):
        xu = synth.fill_host(nu, synth.F32, synth.key(5, synth.KIND_MASTER, 0, 0, u), 0.01)
        # the gathers before the update placed the cast initial weights
        assert d["seen%d" % u].tobytes() == oracle.cast(xu, oracle.BF16).tobytes()
        gu = synth.fill_host(nu, synth.BF16, synth.key(5, synth.KIND_GRAD, 1, 0, u), 1e-3)
        mu, vu = np.zeros(nu, np.float32), np.zeros(nu, np.float32)
        fu = np.zeros(nu, np.uint16)
        oracle.zero_step([gu], oracle.BF16, nu, xu, mu, vu, fu, oracle.BF16, 1e-3, 0.9, 0.999,
                         1e-8, 1)
        xs.append(xu)
        ps.append(fu)
    assert tuple(d["verdict3"]) == (False, False)
    assert d["x3"].tobytes() == np.concatenate(xs).tobytes()
    assert d["p3"].tobytes() == np.concatenate(ps).tobytes()
    assert bool(d["async_ok"])


def test_sharded_step_with_decoupled_weight_decay(tmp_path):
    """AdamW (weight decay 0.1) through ShardedStep and LibraryRank, two
    processes, a skipped step: bit-identical to the oracle's all-ranks
    AdamW step."""
    import oracle
    import synth
    world, numel, inject_at, wd = 2, 200_003, (2, 0, 150_001), 0.1
    mp.start_processes(_rank, args=(world, _free_port(), numel, inject_at, True, str(tmp_path),
                                    wd), nprocs=world, join=True, start_method="spawn")
    S = oracle.shard_size(numel, world)
    P = S * world
    x = np.zeros(P, np.float32)
    x[:numel] = synth.fill_host(numel, synth.F32, synth.key(0, synth.KIND_MASTER), 0.01)
    m, v = np.zeros(P, np.float32), np.zeros(P, np.float32)
    full = np.zeros(P, np.uint16)
    scale, good, t, skips = 2.0 ** 12, 0, 0, []
    for it in (1, 2, 3):
        grads = [synth.fill_host(numel, synth.F16, synth.key(0, synth.KIND_GRAD, it, k),
                                 1e-3 * scale) for k in range(world)]
        if it == inject_at[0]:
            grads[inject_at[1]][inject_at[2]] = 0x7C00
        skipped, _ = oracle.zero_step(grads, oracle.F16, numel, x, m, v, full, oracle.F16, 1e-3,
                                      0.9, 0.999, 1e-8, t + 1, loss_scale=scale,
                                      weight_decay=wd)
        skips.append(skipped)
        if not skipped:
            t += 1
        scale, good = oracle.scale_update(scale, skipped, good, 2000)
    assert skips == [False, True, False]
    for r in range(world):
        d = np.load(os.path.join(tmp_path, "rank%d.npz" % r))
        assert list(d["skips"]) == skips
        sl = slice(r * S, (r + 1) * S)
        assert d["x"].tobytes() == x[sl].tobytes() and d["m"].tobytes() == m[sl].tobytes()
        assert d["v"].tobytes() == v[sl].tobytes() and d["full"].tobytes() == full.tobytes()


@pytest.mark.parametrize("bucket", [0, 50_001])
def test_sharded_stage1_keeps_the_averaged_gradient(tmp_path, bucket):
    """Stage 1 across two processes: besides the step (bit-identical to the
    oracle), every rank ends with the whole averaged gradient of the last
    step -- its own range written by the step, the rest all-gathered --
    equal to the oracle's all-reduce mean (reading: before unscaling, in the
    gradient type)."""
    import oracle
    import synth
    world, numel = 2, 200_003
    mp.start_processes(_rank, args=(world, _free_port(), numel, None, True, str(tmp_path), 0.0,
                                    bucket, 1), nprocs=world, join=True, start_method="spawn")
    x, m, v, full, skips = _all_ranks_reference(numel, world, None)
    S = oracle.shard_size(numel, world)
    P = S * world
    scale = 2.0 ** 12                       # no skip: the scale in force at step 3
    grads = [synth.fill_host(numel, synth.F16, synth.key(0, synth.KIND_GRAD, 3, k), 1e-3 * scale)
             for k in range(world)]
    want = oracle.cast(oracle.all_reduce_mean(grads, oracle.F16, numel), oracle.F16)
    assert want.size == P and not want[numel:].any()     # the padding's mean is +0
    for r in range(world):
        d = np.load(os.path.join(tmp_path, "rank%d.npz" % r))
        sl = slice(r * S, (r + 1) * S)
        assert d["x"].tobytes() == x[sl].tobytes() and d["full"].tobytes() == full.tobytes()
        assert d["avg"].tobytes() == want.tobytes(), r

