"""Oracle-side references for the GPU parity tests.

Everything here is computed by ``oracle`` from inputs drawn on the host by
``synth`` with the same recipe the GPU runner uses on the device
(workloads.runner); nothing is read back from the CUDA path.
"""
from __future__ import annotations

import numpy as np

import oracle
import synth
from workloads import KIND_SHARD, Workload, grad_sigma

STORAGE = oracle.NP_STORAGE


def valid_len(numel, S, rank):
    return max(0, min(S, numel - rank * S))


def host_grads(w: Workload, it: int, scale: float, unit: int = 0):
    """Rank k's local grads at iteration `it` (all-ranks view): numel each."""
    n = w.units[unit] if w.units else w.numel
    sigma = grad_sigma(w, scale)
    out = [synth.fill_host(n, w.grad_dtype, synth.key(w.seed, synth.KIND_GRAD, it, k, unit),
                           sigma) for k in range(w.world)]
    if w.inject and w.inject[0] == it and unit == 0:
        k = w.inject[1]
        e = synth.pick_index(w.seed, n, step=it, rank=k, unit=unit)
        out[k][e] = oracle.cast(np.array([np.inf], np.float32), w.grad_dtype)[0]
    return out


def shard_of(w: Workload, unit: int = 0) -> int:
    return w.unit_shard(unit) if w.units else w.shard


def host_slices(w: Workload, it: int, scale: float, rank: int, unit: int = 0):
    """The S-element slices rank `rank` receives (one-rank view)."""
    n = w.units[unit] if w.units else w.numel
    S = shard_of(w, unit)
    nv = valid_len(n, S, rank)
    sigma = grad_sigma(w, scale)
    out = []
    for k in range(w.world):
        s = np.zeros(S, STORAGE[w.grad_dtype])
        s[:nv] = synth.fill_host(nv, w.grad_dtype,
                                 synth.key(w.seed, synth.KIND_GRAD, it, k, unit), sigma,
                                 index0=rank * S)
        out.append(s)
    if w.inject and w.inject[0] == it and unit == 0:
        k = w.inject[1]
        e = synth.pick_index(w.seed, n, step=it, rank=k, unit=unit)
        if rank * S <= e < rank * S + S:
            out[k][e - rank * S] = oracle.cast(np.array([np.inf], np.float32), w.grad_dtype)[0]
    return out


def host_master(w: Workload, unit: int = 0, rank: int = -1):
    n = w.units[unit] if w.units else w.numel
    S = shard_of(w, unit)
    k = synth.key(w.seed, synth.KIND_MASTER, 0, 0, unit)
    if rank < 0:
        x = np.zeros(S * w.world, np.float32)
        x[:n] = synth.fill_host(n, synth.F32, k, w.sigma_master)
    else:
        x = np.zeros(S, np.float32)
        nv = valid_len(n, S, rank)
        x[:nv] = synth.fill_host(nv, synth.F32, k, w.sigma_master, index0=rank * S)
    return x


def host_other_shard(w: Workload, k: int, unit: int = 0):
    n = w.units[unit] if w.units else w.numel
    S = shard_of(w, unit)
    s = np.zeros(S, STORAGE[w.param_dtype])
    nv = valid_len(n, S, k)
    s[:nv] = synth.fill_host(nv, w.param_dtype, synth.key(w.seed, KIND_SHARD, 0, k, unit),
                             w.sigma_master, index0=k * S)
    return s


class OracleRun:
    """The oracle stepping the same workload (sizes it finishes quickly)."""

    def __init__(self, w: Workload):
        self.w = w
        self.scale = w.loss_scale
        self.good = 0
        self.t = 0
        self.skips = []
        self.gathers = []     # stage 3: unit buffers seen at each gather
        units = range(len(w.units)) if w.units else [0]
        self.state = {}
        for u in units:
            x = host_master(w, u, w.rank)
            self.state[u] = [x, np.zeros_like(x), np.zeros_like(x)]
        if w.stage < 3:
            P = w.shard * w.world
            self.full = np.zeros(P, STORAGE[w.param_dtype])
            if w.rank < 0:
                self.full[:] = oracle.cast(self.state[0][0], w.param_dtype)
            else:
                S = w.shard
                self.full[w.rank * S:(w.rank + 1) * S] = oracle.cast(self.state[0][0],
                                                                     w.param_dtype)
        else:
            self.own = {u: oracle.cast(self.state[u][0], w.param_dtype) for u in units}

    def _unit_shards(self, u):
        w = self.w
        if w.rank < 0:
            return np.split(self.own[u], w.world)
        return [self.own[u] if k == w.rank else host_other_shard(w, k, u)
                for k in range(w.world)]

    def step(self, it: int):
        w = self.w
        t = self.t + 1
        hp = (w.lr, w.beta1, w.beta2, w.eps, t)
        if w.stage < 3:
            x, m, v = self.state[0]
            if w.rank < 0:
                grads = host_grads(w, it, self.scale)
                skipped, _ = oracle.zero_step(grads, w.grad_dtype, w.numel, x, m, v, self.full,
                                              w.param_dtype, *hp, loss_scale=self.scale,
                                              weight_decay=w.weight_decay)
            else:
                S = w.shard
                sl = host_slices(w, it, self.scale, w.rank)
                lp = self.full[w.rank * S:(w.rank + 1) * S].copy()
                skipped, _ = oracle.zero_rank_step(sl, w.grad_dtype, w.numel, w.rank, x, m, v,
                                                   lp, w.param_dtype, *hp,
                                                   loss_scale=self.scale,
                                                   weight_decay=w.weight_decay)
                self.full[w.rank * S:(w.rank + 1) * S] = lp
                if w.gather_after:
                    shards = [lp if k == w.rank else host_other_shard(w, k)
                              for k in range(w.world)]
                    self.full = oracle.all_gather(shards, w.param_dtype)
        else:
            nunits = len(w.units)
            for u in range(nunits):
                self.gathers.append(("fwd", u, oracle.all_gather(self._unit_shards(u),
                                                                 w.param_dtype)))
            new_state, new_own, skipped = {}, {}, False
            for u in reversed(range(nunits)):
                self.gathers.append(("bwd", u, oracle.all_gather(self._unit_shards(u),
                                                                 w.param_dtype)))
                x, m, v = [a.copy() for a in self.state[u]]
                if w.rank < 0:
                    grads = host_grads(w, it, self.scale, u)
                    full = np.zeros(x.size, STORAGE[w.param_dtype])
                    sk, _ = oracle.zero_step(grads, w.grad_dtype, w.units[u], x, m, v, full,
                                             w.param_dtype, *hp, loss_scale=self.scale,
                                             weight_decay=w.weight_decay,
                                             shard=w.unit_shard(u))
                    lp = full
                else:
                    sl = host_slices(w, it, self.scale, w.rank, u)
                    lp = self.own[u].copy()
                    sk, _ = oracle.zero_rank_step(sl, w.grad_dtype, w.units[u], w.rank, x, m,
                                                  v, lp, w.param_dtype, *hp,
                                                  loss_scale=self.scale,
                                                  weight_decay=w.weight_decay,
                                                  shard=w.unit_shard(u))
                skipped |= sk
                new_state[u] = [x, m, v]
                new_own[u] = lp
            if not skipped:
                self.state.update(new_state)
                self.own.update(new_own)
        self.skips.append(bool(skipped))
        if not skipped:
            self.t += 1
        if self.scale > 0:
            self.scale, self.good = oracle.scale_update(self.scale, skipped, self.good,
                                                        w.growth_interval)
        return skipped


def sampled_reference(w: Workload, idx: np.ndarray, iterations, skipped_iters=(), rank=-1,
                      unit: int = 0):
    """Oracle state at flat positions `idx` after the given iterations, one
    element at a time (the update is elementwise).  Positions index the
    bound state: the all-ranks flat vector (rank = -1) or rank `rank`'s
    shard.  The global skip verdicts are given (`skipped_iters`).  Returns
    (master, m, v, param) at idx."""
    n = w.units[unit] if w.units else w.numel
    S = shard_of(w, unit)
    gidx = idx if rank < 0 else idx + rank * S      # global flat position
    valid = gidx < n
    kmaster = synth.key(w.seed, synth.KIND_MASTER, 0, 0, unit)
    x = np.zeros(idx.size, np.float32)
    x[valid] = synth.fill_host(int(valid.sum()), synth.F32, kmaster, w.sigma_master,
                               indices=gidx[valid])
    m = np.zeros_like(x)
    v = np.zeros_like(x)
    scale, good, t = w.loss_scale, 0, 0
    for it in iterations:
        skipped = it in skipped_iters
        if not skipped:
            t += 1
            sigma = grad_sigma(w, scale)
            bufs = []
            for k in range(w.world):
                b = np.zeros(idx.size, STORAGE[w.grad_dtype])
                b[valid] = synth.fill_host(int(valid.sum()), w.grad_dtype,
                                           synth.key(w.seed, synth.KIND_GRAD, it, k, unit),
                                           sigma, indices=gidx[valid])
                bufs.append(b)
            acc = oracle.rank_sum(bufs, w.grad_dtype, idx.size, idx.size)
            g, _ = oracle.average(acc, w.world, scale)
            oracle.adam(x, m, v, g, w.lr, w.beta1, w.beta2, w.eps, t,
            weight_decay=w.weight_decay)
        if scale > 0:
            scale, good = oracle.scale_update(scale, skipped, good, w.growth_interval)
    return x, m, v, oracle.cast(x, w.param_dtype)
