"""The multi-rank protocol on CPU with real collectives (gloo, 2 and 4
processes): each process is one data-parallel rank in the one-rank view,
driven by the library's sharded step (zero_sharded_optimizer_step_gb300.
sharded: the all-to-all of the grad slices, the overflow verdict combined
across ranks with a MAX all-reduce between the local pass and the rest of
the step, the all-gather of the cast shards) with the rank's arithmetic done
by the oracle -- and the result must be bit-identical to the all-ranks step.  The same for ZeRO-3:
per unit an all-gather before forward and backward, the unit's
reduce-scatter, and every unit's verdict combined before any unit's Adam
counts.  Also covers the benchmark's cross-rank timing helpers (barrier,
max over ranks)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleRank:
    """Rank `rank`'s own arithmetic done by the CPU oracle, with the members
    the library's ShardedStep drives (the same ones LibraryRank has): fp16
    grads and params held as 16-bit patterns in CPU tensors, the step-tagged
    flag word, the oracle's one-rank step once the verdict is combined."""

    def __init__(self, numel, world, rank, params=None, flag=None):
        import oracle
        import synth
        self.oracle = oracle
        self.numel, self.world, self.rank = numel, world, rank
        self.shard = S = oracle.shard_size(numel, world)
        lo = rank * S
        self.nv = max(0, min(S, numel - lo))
        self.x = np.zeros(S, np.float32)
        self.x[:self.nv] = synth.fill_host(self.nv, synth.F32, synth.key(0, synth.KIND_MASTER),
                                           0.01, index0=lo)
        self.m, self.v = np.zeros(S, np.float32), np.zeros(S, np.float32)
        # the ranks of one process may share the parameter buffer and the flag
        self.params = torch.zeros(S * world, dtype=torch.int16) if params is None else params
        self.own_params = self.params[lo:lo + S]
        self.own_params.copy_(torch.from_numpy(oracle.cast(self.x, oracle.F16).view(np.int16)))
        self.flag = torch.zeros(1, dtype=torch.int64) if flag is None else flag
        self.step_id = 0

    def grad_buffer(self, n):
        return torch.zeros(n, dtype=torch.int16)

    def local_pass(self, slices, lr, beta1, beta2, eps, t, loss_scale):
        o = self.oracle
        self.step_id += 1
        self.scale = loss_scale
        self.sl = [s.numpy().view(np.uint16).copy() for s in slices]
        acc = o.rank_sum(self.sl, o.F16, self.shard, self.nv)
        _, bad = o.average(acc, self.world, loss_scale)
        if bad:
            self.flag[0] = self.step_id

    def finish(self, lr, beta1, beta2, eps, t):
        o = self.oracle
        others = int(self.flag.item() == self.step_id)     # any rank's finding
        lp = self.own_params.numpy().view(np.uint16).copy()
        o.zero_rank_step(self.sl, o.F16, self.numel, self.rank, self.x, self.m, self.v, lp,
                         o.F16, lr, beta1, beta2, eps, t, loss_scale=self.scale,
                         others_nonfinite=others)
        self.own_params.copy_(torch.from_numpy(lp.view(np.int16)))

    def status(self):
        bad = self.flag.item() == self.step_id
        return bad, bad and self.scale > 0

    # the bucketed form: pieces of the shard arrive bucket by bucket; each
    # piece's local verdict at once, the oracle's step on the whole shard once
    # the combined verdict is in (the update is elementwise)
    def bucket_begin(self, loss_scale):
        self.step_id += 1
        self.scale = loss_scale
        self.sl = [np.zeros(self.shard, np.uint16) for _ in range(self.world)]

    def bucket_pass(self, offset, count, slices, lr, beta1, beta2, eps, t):
        o = self.oracle
        piece = []
        for k, s in enumerate(slices):
            self.sl[k][offset:offset + count] = s.numpy().view(np.uint16)
            piece.append(self.sl[k][offset:offset + count].copy())
        nv = max(0, min(count, self.nv - offset))
        _, bad = o.average(o.rank_sum(piece, o.F16, count, nv), self.world, self.scale)
        if bad:
            self.flag[0] = self.step_id

    def bucket_end(self, lr, beta1, beta2, eps, t):
        self.finish(lr, beta1, beta2, eps, t)


def _rank_main(rank, world, port, numel, inject_at, out_dir, bucket=0):
    """One data-parallel rank, driven by the library's sharded step (the
    all-to-all of the grad slices, the MAX combine of the flag word, the
    all-gather of the cast shards) with the oracle's arithmetic."""
    import sys
    sys.path.insert(0, ROOT)
    import oracle
    import synth
    from zero_sharded_optimizer_step_gb300.sharded import ShardedStep
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local = OracleRank(numel, world, rank)
    step = ShardedStep(local)
    P = local.shard * world
    scale, good, t = 2.0 ** 12, 0, 0
    skips = []
    for it in (1, 2, 3):
        g = np.zeros(P, np.uint16)
        g[:numel] = synth.fill_host(numel, synth.F16, synth.key(0, synth.KIND_GRAD, it, rank),
                                    1e-3 * scale)
        if inject_at and it == inject_at[0] and rank == inject_at[1]:
            g[inject_at[2]] = 0x7C00                          # +inf in fp16
        gt = torch.from_numpy(g.view(np.int16))
        if bucket:
            # the same step bucket by bucket, each bucket from one reused buffer
            buf = torch.zeros(bucket, dtype=torch.int16)
            step.begin(scale)
            for off in range(0, P, bucket):
                n = min(bucket, P - off)
                buf[:n].copy_(gt[off:off + n])
                step.bucket(off, buf[:n], 1e-3, 0.9, 0.999, 1e-8, t + 1)
            _, skipped = step.end(1e-3, 0.9, 0.999, 1e-8, t + 1)
        else:
            _, skipped = step.step(gt, 1e-3, 0.9, 0.999, 1e-8, t + 1, loss_scale=scale)
        skips.append(skipped)
        if not skipped:
            t += 1
        scale, good = oracle.scale_update(scale, skipped, good, 2000)
    full = local.params.numpy().view(np.uint16)
    np.savez(os.path.join(out_dir, "rank%d.npz" % rank), x=local.x, m=local.m, v=local.v,
             full=full, skips=np.array(skips))
    # the benchmark's helpers under gloo
    sys.argv = ["bench.py"]
    import bench
    bench.barrier(world)
    assert bench.allreduce_max(float(rank) * 1.5, world) == 1.5 * (world - 1)
    dist.destroy_process_group()


def _all_ranks_reference(numel, world, inject_at):
    import oracle
    import synth
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
        if inject_at and it == inject_at[0]:
            grads[inject_at[1]][inject_at[2]] = 0x7C00
        skipped, _ = oracle.zero_step(grads, oracle.F16, numel, x, m, v, full, oracle.F16,
                                      1e-3, 0.9, 0.999, 1e-8, t + 1, loss_scale=scale)
        skips.append(skipped)
        if not skipped:
            t += 1
        scale, good = oracle.scale_update(scale, skipped, good, 2000)
    return x, m, v, full, skips


@pytest.mark.parametrize("world,numel,inject_at,bucket", [
    (2, 10_001, None, 0),
    (2, 10_001, (2, 1, 9_999), 0),      # rank 1's element in rank 1's shard
    (4, 20_003, (2, 3, 17), 0),         # rank 3's element in rank 0's shard
    (2, 10_001, (2, 1, 9_999), 3_001),  # buckets, one across the shard boundary
    (4, 20_003, (2, 3, 17), 7_000),
    (4, 20_003, None, 20_004),          # one bucket: the whole vector
    (3, 10_001, (2, 2, 5), 2_500),      # three ranks, one pad element, odd buckets
])
def test_one_rank_views_with_real_collectives(tmp_path, world, numel, inject_at, bucket):
    port = _free_port()
    mp.start_processes(_rank_main, args=(world, port, numel, inject_at, str(tmp_path), bucket),
                       nprocs=world, join=True, start_method="spawn")
    import oracle
    x, m, v, full, skips = _all_ranks_reference(numel, world, inject_at)
    S = oracle.shard_size(numel, world)
    want_skips = [bool(inject_at) and it == inject_at[0] for it in (1, 2, 3)]
    assert skips == want_skips
    for r in range(world):
        d = np.load(os.path.join(tmp_path, "rank%d.npz" % r))
        assert list(d["skips"]) == skips, r
        sl = slice(r * S, (r + 1) * S)
        assert d["x"].tobytes() == x[sl].tobytes()
        assert d["m"].tobytes() == m[sl].tobytes()
        assert d["v"].tobytes() == v[sl].tobytes()
        assert d["full"].tobytes() == full.tobytes()


class OracleRanks:
    """The view of k consecutive ranks (the members RanksStep drives, as the
    library's LibraryRank(n_ranks=k) has them), each rank's arithmetic done
    by the oracle: its pieces of k*S elements are cut into the k ranks'
    slices; one parameter buffer and one flag word for all."""

    def __init__(self, numel, world, first, k):
        import oracle
        self.n_ranks, self.rank = k, first
        self.shard = S = oracle.shard_size(numel, world)
        self.params = torch.zeros(S * world, dtype=torch.int16)
        self.flag = torch.zeros(1, dtype=torch.int64)
        self.ranks = [OracleRank(numel, world, first + j, self.params, self.flag)
                      for j in range(k)]
        self.own_params = self.params[first * S:(first + k) * S]

    def grad_buffer(self, n):
        return torch.zeros(n, dtype=torch.int16)

    def local_pass(self, pieces, lr, beta1, beta2, eps, t, loss_scale):
        S = self.shard
        for j, r in enumerate(self.ranks):
            r.local_pass([pc[j * S:(j + 1) * S] for pc in pieces], lr, beta1, beta2, eps, t,
                         loss_scale)

    def finish(self, lr, beta1, beta2, eps, t):
        for r in self.ranks:
            r.finish(lr, beta1, beta2, eps, t)

    def status(self):
        return self.ranks[0].status()


def _ranks_main(proc, nprocs, port, numel, world, inject_at, out_dir):
    """Process `proc` of `nprocs` holding world // nprocs consecutive ranks
    in one view (RanksStep), each rank's arithmetic the oracle's."""
    import sys
    sys.path.insert(0, ROOT)
    import oracle
    import synth
    from zero_sharded_optimizer_step_gb300.sharded import RanksStep
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=proc, world_size=nprocs)
    k = world // nprocs
    S = oracle.shard_size(numel, world)
    P = S * world
    view = OracleRanks(numel, world, proc * k, k)
    params, ranks = view.params, view.ranks
    step = RanksStep(view)
    scale, good, t, skips = 2.0 ** 12, 0, 0, []
    for it in (1, 2, 3):
        gts = []
        for c in range(k):
            r = proc * k + c
            g = np.zeros(P, np.uint16)
            g[:numel] = synth.fill_host(numel, synth.F16, synth.key(0, synth.KIND_GRAD, it, r),
                                        1e-3 * scale)
            if inject_at and it == inject_at[0] and r == inject_at[1]:
                g[inject_at[2]] = 0x7C00
            gts.append(torch.from_numpy(g.view(np.int16)))
        _, skipped = step.step(gts, 1e-3, 0.9, 0.999, 1e-8, t + 1, loss_scale=scale)
        skips.append(skipped)
        if not skipped:
            t += 1
        scale, good = oracle.scale_update(scale, skipped, good, 2000)
    for c, r in enumerate(ranks):
        np.savez(os.path.join(out_dir, "rank%d.npz" % r.rank), x=r.x, m=r.m, v=r.v,
                 full=params.numpy().view(np.uint16), skips=np.array(skips))
    dist.destroy_process_group()


@pytest.mark.parametrize("nprocs,world,numel,inject_at", [
    (1, 4, 20_003, (2, 3, 17)),          # all four ranks in one process: no collective
    (2, 4, 20_003, (2, 3, 17)),          # two ranks per process
    (2, 4, 10_001, (2, 1, 9_999)),       # one pad element, the planted value in rank 3's shard
    (2, 6, 10_001, None),
    (3, 6, 10_001, (2, 4, 5)),           # three processes of two ranks
])
def test_ranks_per_process_with_real_collectives(tmp_path, nprocs, world, numel, inject_at):
    port = _free_port()
    mp.start_processes(_ranks_main, args=(nprocs, port, numel, world, inject_at, str(tmp_path)),
                       nprocs=nprocs, join=True, start_method="spawn")
    import oracle
    x, m, v, full, skips = _all_ranks_reference(numel, world, inject_at)
    S = oracle.shard_size(numel, world)
    assert skips == [bool(inject_at) and it == inject_at[0] for it in (1, 2, 3)]
    for r in range(world):
        d = np.load(os.path.join(tmp_path, "rank%d.npz" % r))
        assert list(d["skips"]) == skips, r
        sl = slice(r * S, (r + 1) * S)
        assert d["x"].tobytes() == x[sl].tobytes(), r
        assert d["m"].tobytes() == m[sl].tobytes(), r
        assert d["v"].tobytes() == v[sl].tobytes(), r
        assert d["full"].tobytes() == full.tobytes(), r


# ------------------------------------------------------------------ stage 3

class OracleRank3:
    """Rank `rank`'s own arithmetic of a stage-3 step done by the CPU oracle,
    with the members the library's ShardedZero3Step drives (LibraryRank3's):
    per unit fp16 param shards as 16-bit patterns in CPU tensors, the
    step-tagged flag word; each unit's local verdict at its pass, every
    unit's Adam once the combined verdict is in."""

    def __init__(self, units, world, rank):
        import oracle
        import synth
        self.o = oracle
        self.units, self.world, self.rank = list(units), world, rank
        self.shards = [oracle.shard_size(nu, world) for nu in units]
        self.state, self.lp = [], []
        for u, (nu, S) in enumerate(zip(units, self.shards)):
            nv = max(0, min(S, nu - rank * S))
            x = np.zeros(S, np.float32)
            x[:nv] = synth.fill_host(nv, synth.F32, synth.key(0, synth.KIND_MASTER, 0, 0, u),
                                     0.01, index0=rank * S)
            self.state.append([x, np.zeros(S, np.float32), np.zeros(S, np.float32)])
            self.lp.append(torch.from_numpy(oracle.cast(x, oracle.F16).view(np.int16)).clone())
        self.flag = torch.zeros(1, dtype=torch.int64)
        self.step_id = 0

    def grad_buffer(self, n):
        return torch.zeros(n, dtype=torch.int16)

    def param_buffer(self, n):
        return torch.zeros(n, dtype=torch.int16)

    def own_params(self, u):
        return self.lp[u]

    def begin(self, loss_scale):
        self.step_id += 1
        self.scale = loss_scale
        self.pending = {}

    def unit_pass(self, u, slices, lr, beta1, beta2, eps, t, loss_scale):
        o = self.o
        S = self.shards[u]
        nv = max(0, min(S, self.units[u] - self.rank * S))
        sl = [s.numpy().view(np.uint16).copy() for s in slices]
        _, bad = o.average(o.rank_sum(sl, o.F16, S, nv), self.world, loss_scale)
        if bad:
            self.flag[0] = self.step_id
        self.pending[u] = sl

    def finish(self, lr, beta1, beta2, eps, t):
        o = self.o
        others = int(self.flag.item() == self.step_id)    # any unit on any rank
        for u, sl in self.pending.items():
            x, m, v = self.state[u]
            lp = self.lp[u].numpy().view(np.uint16).copy()
            o.zero_rank_step(sl, o.F16, self.units[u], self.rank, x, m, v, lp, o.F16, lr,
                             beta1, beta2, eps, t, loss_scale=self.scale,
                             others_nonfinite=others)
            self.lp[u].copy_(torch.from_numpy(lp.view(np.int16)))

    def status(self):
        bad = self.flag.item() == self.step_id
        return bad, bad and self.scale > 0


def _rank_main3(rank, world, port, units, inject_at, out_dir, prefetch=False):
    """One rank of a ZeRO-3 step over gloo through the library's
    ShardedZero3Step: per unit an all-gather of the cast shards before
    forward and again before backward, the unit's grads exchanged after its
    backward (here: the seeded draws), every unit's verdict combined (MAX)
    before any unit's Adam counts."""
    import sys
    sys.path.insert(0, ROOT)
    import oracle
    import synth
    from zero_sharded_optimizer_step_gb300.sharded import ShardedZero3Step
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local = OracleRank3(units, world, rank)
    step = ShardedZero3Step(local, prefetch=prefetch)
    scale, good, t, skips, gathered, seen = 2.0 ** 12, 0, 0, [], {}, []
    for it in (1, 2, 3):
        def forward(u, params):
            seen.append(("fwd", u))
            gathered[u] = params.numpy().view(np.uint16).copy()

        def backward(u, params):
            seen.append(("bwd", u))
            gathered[u] = params.numpy().view(np.uint16).copy()
            nu, S = units[u], local.shards[u]
            g = np.zeros(S * world, np.uint16)
            g[:nu] = synth.fill_host(nu, synth.F16, synth.key(0, synth.KIND_GRAD, it, rank, u),
                                     1e-3 * scale)
            if inject_at and (it, rank, u) == inject_at[:3]:
                g[inject_at[3]] = 0x7C00                  # +inf in fp16
            return torch.from_numpy(g.view(np.int16))
        _, skipped = step.step(backward, 1e-3, 0.9, 0.999, 1e-8, t + 1, loss_scale=scale,
                               forward=forward)
        skips.append(skipped)
        if not skipped:
            t += 1
        scale, good = oracle.scale_update(scale, skipped, good, 2000)
    U = len(units)
    assert seen == 3 * ([("fwd", u) for u in range(U)] + [("bwd", u) for u in reversed(range(U))])
    out = {"skips": np.array(skips)}
    for u in range(U):
        out["x%d" % u], out["m%d" % u], out["v%d" % u] = local.state[u]
        out["lp%d" % u] = local.lp[u].numpy().view(np.uint16)
        out["full%d" % u] = gathered[u]
    np.savez(os.path.join(out_dir, "rank%d.npz" % rank), **out)
    dist.destroy_process_group()


class OracleRanks3:
    """The view of k consecutive ranks of a stage-3 step (the members
    ShardedZero3Step drives, as LibraryRank3(n_ranks=k) has them), each
    rank's arithmetic the oracle's (OracleRank3): per unit the k ranks'
    param shards end to end in one tensor, one flag word for all; with every
    rank held, `place` is the gather."""

    def __init__(self, units, world, first, k):
        self.n_ranks, self.rank, self.world = k, first, world
        self.subs = [OracleRank3(units, world, first + j) for j in range(k)]
        self.shards = self.subs[0].shards
        self.flag = torch.zeros(1, dtype=torch.int64)
        self.lp = []
        for u, S in enumerate(self.shards):
            joined = torch.cat([s.lp[u] for s in self.subs])
            self.lp.append(joined)
            for j, s in enumerate(self.subs):
                s.lp[u] = joined[j * S:(j + 1) * S]      # each rank writes its part in place
        for s in self.subs:
            s.flag = self.flag

    def grad_buffer(self, n):
        return torch.zeros(n, dtype=torch.int16)

    def param_buffer(self, n):
        return torch.zeros(n, dtype=torch.int16)

    def own_params(self, u):
        return self.lp[u]

    def place(self, u, full):
        assert self.n_ranks == self.world
        full.copy_(self.lp[u])

    def begin(self, loss_scale):
        for s in self.subs:
            s.begin(loss_scale)

    def unit_pass(self, u, pieces, lr, beta1, beta2, eps, t, loss_scale):
        S = self.shards[u]
        for j, s in enumerate(self.subs):
            s.unit_pass(u, [pc[j * S:(j + 1) * S] for pc in pieces], lr, beta1, beta2, eps, t,
                        loss_scale)

    def finish(self, lr, beta1, beta2, eps, t):
        for s in self.subs:
            s.finish(lr, beta1, beta2, eps, t)

    def status(self):
        return self.subs[0].status()


def _ranks_main3(proc, nprocs, port, world, units, inject_at, out_dir, prefetch):
    """Process `proc` of `nprocs` holding world // nprocs consecutive ranks of
    a ZeRO-3 step (ShardedZero3Step over a view of several ranks)."""
    import sys
    sys.path.insert(0, ROOT)
    import oracle
    import synth
    from zero_sharded_optimizer_step_gb300.sharded import ShardedZero3Step
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=proc, world_size=nprocs)
    k = world // nprocs
    view = OracleRanks3(units, world, proc * k, k)
    step = ShardedZero3Step(view, prefetch=prefetch)
    scale, good, t, skips, gathered = 2.0 ** 12, 0, 0, [], {}
    for it in (1, 2, 3):
        def backward(u, params):
            gathered[u] = params.numpy().view(np.uint16).copy()
            nu, S = units[u], view.shards[u]
            out = []
            for c in range(k):
                r = proc * k + c
                g = np.zeros(S * world, np.uint16)
                g[:nu] = synth.fill_host(nu, synth.F16, synth.key(0, synth.KIND_GRAD, it, r, u),
                                         1e-3 * scale)
                if inject_at and (it, r, u) == inject_at[:3]:
                    g[inject_at[3]] = 0x7C00
                out.append(torch.from_numpy(g.view(np.int16)))
            return out
        _, skipped = step.step(backward, 1e-3, 0.9, 0.999, 1e-8, t + 1, loss_scale=scale)
        skips.append(skipped)
        if not skipped:
            t += 1
        scale, good = oracle.scale_update(scale, skipped, good, 2000)
    for j, s in enumerate(view.subs):
        out = {"skips": np.array(skips)}
        for u in range(len(units)):
            out["x%d" % u], out["m%d" % u], out["v%d" % u] = s.state[u]
            out["lp%d" % u] = s.lp[u].numpy().view(np.uint16)
            out["full%d" % u] = gathered[u]
        np.savez(os.path.join(out_dir, "rank%d.npz" % (proc * k + j)), **out)
    dist.destroy_process_group()


def _stage3_reference(units, world, inject_at):
    """All ranks in one process: per unit the oracle's all-ranks step on the
    unit's own flat vector; a step counts only if no unit overflowed."""
    import oracle
    import synth
    st, fulls = [], []
    for u, nu in enumerate(units):
        P = oracle.shard_size(nu, world) * world
        x = np.zeros(P, np.float32)
        x[:nu] = synth.fill_host(nu, synth.F32, synth.key(0, synth.KIND_MASTER, 0, 0, u), 0.01)
        st.append([x, np.zeros(P, np.float32), np.zeros(P, np.float32)])
        fulls.append(oracle.cast(x, oracle.F16))
    scale, good, t, skips = 2.0 ** 12, 0, 0, []
    for it in (1, 2, 3):
        new, skipped = [], False
        for u, nu in enumerate(units):
            grads = [synth.fill_host(nu, synth.F16, synth.key(0, synth.KIND_GRAD, it, k, u),
                                     1e-3 * scale) for k in range(world)]
            if inject_at and (it, u) == (inject_at[0], inject_at[2]):
                grads[inject_at[1]][inject_at[3]] = 0x7C00
            x, m, v = (a.copy() for a in st[u])
            full = fulls[u].copy()
            sk, _ = oracle.zero_step(grads, oracle.F16, nu, x, m, v, full, oracle.F16, 1e-3, 0.9,
                                     0.999, 1e-8, t + 1, loss_scale=scale)
            skipped = skipped or sk
            new.append(([x, m, v], full))
        if not skipped:
            st = [n[0] for n in new]
            fulls = [n[1] for n in new]
            t += 1
        skips.append(skipped)
        scale, good = oracle.scale_update(scale, skipped, good, 2000)
    return st, fulls, skips


@pytest.mark.parametrize("world,units,inject_at,prefetch", [
    (2, [3001, 17, 5000], None, False),
    (2, [3001, 17, 5000], (2, 1, 0, 1400), False),    # (iteration, rank, unit, element)
    (4, [3001, 17, 5000], (2, 3, 2, 11), False),     # rank 3's element in rank 0's shard of unit 2
    (2, [3001, 17, 5000, 64], (2, 1, 0, 1400), True),  # the next unit's gather in flight
    (4, [3001, 17, 5000], (2, 3, 2, 11), True),
    (3, [3001, 17, 5000], (2, 2, 1, 16), True),     # three ranks: padding in every unit
])
def test_stage3_ranks_with_real_collectives(tmp_path, world, units, inject_at, prefetch):
    port = _free_port()
    mp.start_processes(_rank_main3, args=(world, port, units, inject_at, str(tmp_path), prefetch),
                       nprocs=world, join=True, start_method="spawn")
    import oracle
    st, fulls, skips = _stage3_reference(units, world, inject_at)
    assert skips == [bool(inject_at) and it == 2 for it in (1, 2, 3)]
    for r in range(world):
        d = np.load(os.path.join(tmp_path, "rank%d.npz" % r))
        assert list(d["skips"]) == skips, r
        for u, nu in enumerate(units):
            S = oracle.shard_size(nu, world)
            sl = slice(r * S, (r + 1) * S)
            for name, a in zip("xmv", st[u]):
                assert d["%s%d" % (name, u)].tobytes() == a[sl].tobytes(), (r, u, name)
            assert d["lp%d" % u].tobytes() == fulls[u][sl].tobytes()
            # the last gather (before unit u's backward) placed the shards
            # every rank held then, which the third step has since updated
        # every rank saw the same gathered units
        if r == 0:
            first = {u: d["full%d" % u].copy() for u in range(len(units))}
        else:
            for u in range(len(units)):
                assert d["full%d" % u].tobytes() == first[u].tobytes()


@pytest.mark.parametrize("nprocs,world,units,inject_at,prefetch", [
    (1, 4, [3001, 17, 5000], (2, 3, 2, 11), False),    # every rank in one process
    (2, 4, [3001, 17, 5000], (2, 3, 2, 11), False),    # two ranks per process
    (2, 4, [3001, 17, 5000, 64], (2, 1, 0, 1400), True),
    (1, 3, [3001, 17, 5000], (2, 2, 1, 16), True),     # padding in every unit
])
def test_stage3_ranks_per_process(tmp_path, nprocs, world, units, inject_at, prefetch):
    port = _free_port()
    mp.start_processes(_ranks_main3, args=(nprocs, port, world, units, inject_at, str(tmp_path),
                                           prefetch), nprocs=nprocs, join=True,
                       start_method="spawn")
    import oracle
    st, fulls, skips = _stage3_reference(units, world, inject_at)
    assert skips == [bool(inject_at) and it == 2 for it in (1, 2, 3)]
    for r in range(world):
        d = np.load(os.path.join(tmp_path, "rank%d.npz" % r))
        assert list(d["skips"]) == skips, r
        for u, nu in enumerate(units):
            S = oracle.shard_size(nu, world)
            sl = slice(r * S, (r + 1) * S)
            for name, a in zip("xmv", st[u]):
                assert d["%s%d" % (name, u)].tobytes() == a[sl].tobytes(), (r, u, name)
            assert d["lp%d" % u].tobytes() == fulls[u][sl].tobytes()
        if r == 0:
            first = {u: d["full%d" % u].copy() for u in range(len(units))}
        else:
            for u in range(len(units)):
                assert d["full%d" % u].tobytes() == first[u].tobytes()
