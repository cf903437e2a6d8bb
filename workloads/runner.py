"""Runs a Workload on one GPU through the C ABI binding.

PyTorch allocates the buffers; ``synth`` draws the inputs on the device; every
step of the method runs in libzero.so.  Shared by the GPU tests and bench.py.

Index space of the draws (the same on the oracle side): rank k's local
gradient at iteration `it` and flat position i is stream (GRAD, it, k, unit)
at index i; the initial master weight at i is stream (MASTER, 0, 0, unit) at
index i.  In one rank's view rank r holds positions r*S ... r*S+S-1.
"""
from __future__ import annotations

import torch

import synth
import zero_sharded_optimizer_step_gb300 as z

from . import F32, KIND_SHARD, Workload, grad_sigma

TORCH_DTYPE = {0: torch.float32, 1: torch.bfloat16, 2: torch.float16}


def valid_len(numel: int, S: int, rank: int) -> int:
    """Positions of rank `rank`'s shard that hold real parameters."""
    return max(0, min(S, numel - rank * S))


def inject_index(w: Workload, it: int, rank: int, unit: int = 0) -> int:
    n = w.units[unit] if w.units else w.numel
    return synth.pick_index(w.seed, n, step=it, rank=rank, unit=unit)


# Shards from this size on are placed by the row kernel, at the copy rate
# whatever the launch count; a pair's launch saves only on smaller ones.
PAIR_MAX_SHARD_BYTES = 32 << 20


def forward_runs(w: Workload, pairs: bool = True):
    """The stage-3 forward's gather calls over units without groups, each a
    run (first unit, count).  With pairs, two consecutive units whose shards
    are both under PAIR_MAX_SHARD_BYTES are placed by one call into two unit
    buffers ("ZeRO 与 FSDP…", ZeRO-3 与 FSDP: the next unit's all-gather is
    issued before the current unit computes); every other unit alone."""
    U = len(w.units or [])
    es = 4 if w.param_dtype == F32 else 2
    small = [w.unit_shard(u) * es < PAIR_MAX_SHARD_BYTES for u in range(U)]
    runs, u = [], 0
    while u < U:
        if pairs and u + 1 < U and small[u] and small[u + 1]:
            runs.append((u, 2))
            u += 2
        else:
            runs.append((u, 1))
            u += 1
    return runs


def backward_chunks(w: Workload, pairs: bool = True):
    """The stage-3 backward in chunks of two units when every unit is small
    (shards under PAIR_MAX_SHARD_BYTES), from the last unit down: the first
    chunk is gathered, then each call steps a chunk and gathers the next
    (zero3_step_units_gather, two unit buffers) -- the next two units'
    gathers issued while the current two are worked on ("ZeRO 与 FSDP…",
    ZeRO-3 与 FSDP).  None: the unit-by-unit visits instead."""
    U = len(w.units or [])
    es = 4 if w.param_dtype == F32 else 2
    if not pairs or U < 2 or w.groups or any(w.unit_shard(u) * es >= PAIR_MAX_SHARD_BYTES
                                             for u in range(U)):
        return None
    chunks, hi = [], U
    while hi > 0:
        lo = max(0, hi - 2)
        chunks.append((lo, hi - lo))
        hi = lo
    return chunks


class Runner:
    def __init__(self, w: Workload, device: str = "cuda:0", scratch: bool | None = None,
                 shadow: bool = False, alloc_grads: bool = True, hyper: bool = False,
                 visits: str = "fused", fwd_pairs: bool = True):
        self.w = w
        # stage 3 backward: "fused" issues unit u's update and the gather of
        # unit u-1 as one call (zero3_step_unit_gather), "separate" as two
        assert visits in ("fused", "separate")
        self.visits = visits
        # stage 3 over two unit buffers (units without groups): the forward
        # in pairs of small units (forward_runs) and, when every unit is
        # small, the backward in chunks of two (backward_chunks); False:
        # unit by unit, over one unit buffer's worth of schedule
        self.fwd_pairs = fwd_pairs
        self.dev = torch.device(device)
        torch.cuda.set_device(self.dev)
        if w.unit_rows:
            self.ctx = z.zero_init_dim0(w.world, w.grad_dtype, w.param_dtype, w.rank, w.unit_rows)
        else:
            self.ctx = z.zero_init(w.numel, w.world, w.stage, w.grad_dtype, w.param_dtype,
                                   w.rank, w.units)
        ns = z.zero_ctx_state_elems(self.ctx)
        npar = z.zero_ctx_param_elems(self.ctx)
        f32 = dict(dtype=torch.float32, device=self.dev)
        self.master = torch.zeros(ns, **f32)
        self.m = torch.zeros(ns, **f32)
        self.v = torch.zeros(ns, **f32)
        self.params = torch.zeros(npar, dtype=TORCH_DTYPE[w.param_dtype], device=self.dev)
        need_scratch = (w.loss_scale > 0 and not shadow) if scratch is None else scratch
        self.g = torch.zeros(ns, **f32) if need_scratch else None
        self.flag = torch.zeros(1, dtype=torch.int64, device=self.dev)
        z.zero_bind(self.ctx, self.master, self.m, self.v, self.params, self.g, self.flag)
        self.shadow = None
        if shadow:
            # a second state set: every step is one pass, loss-scaled or not
            self.shadow = (torch.zeros(ns, **f32), torch.zeros(ns, **f32),
                           torch.zeros(ns, **f32))
            self.cur = torch.zeros(1, dtype=torch.int64, device=self.dev)
            z.zero_bind_shadow(self.ctx, *self.shadow, self.cur)
        if w.weight_decay:
            z.zero_set_weight_decay(self.ctx, w.weight_decay)
        self.grad_avg = None
        if w.allreduce_out:
            # stage 1: the all-reduced mean grads, P elements of the grad type
            self.grad_avg = torch.zeros(w.shard * w.world, dtype=TORCH_DTYPE[w.grad_dtype],
                                        device=self.dev)
            z.zero_bind_allreduce_out(self.ctx, self.grad_avg)
        self.hyper = None
        if hyper:
            # the per-step scalars from a device block (the form a CUDA graph
            # replays), refreshed before every step
            self.hyper = (torch.zeros(z.ZERO_HYPER_BYTES, dtype=torch.uint8, device=self.dev),
                          torch.zeros(z.ZERO_HYPER_BYTES, dtype=torch.uint8, pin_memory=True))
            z.zero_bind_hyper(self.ctx, self.hyper[0])
        self.stream = torch.cuda.current_stream(self.dev)
        self.scale = w.loss_scale
        self.good = 0
        self.t = 0
        self.skips = []
        self._init_state()
        if alloc_grads:
            self._alloc_grads()
        else:
            self.grads = [[]]     # the caller supplies constant-size bucket buffers
        self._alloc_shards()

    # ------------------------------------------------------------ set-up

    def _fill(self, buf: torch.Tensor, n: int, dtype: int, key: int, sigma: float,
              index0: int = 0):
        if n > 0:
            synth.fill_device(buf.data_ptr(), n, dtype, key, sigma, self.stream.cuda_stream,
                              index0=index0)

    def _units(self):
        """(unit id, numel, S, state offset) for every shardable range."""
        w = self.w
        if w.stage < 3:
            return [(0, w.numel, w.shard, 0)]
        return [(u, w.units[u], w.unit_shard(u), z.zero_ctx_unit_state_offset(self.ctx, u))
                for u in range(len(w.units))]

    def _init_state(self):
        w = self.w
        for u, nu, Su, off in self._units():
            k = synth.key(w.seed, synth.KIND_MASTER, 0, 0, u)
            if w.rank < 0:
                self._fill(self.master[off:], nu, synth.F32, k, w.sigma_master)
            else:
                self._fill(self.master[off:], valid_len(nu, Su, w.rank), synth.F32, k,
                           w.sigma_master, index0=w.rank * Su)
        # the low-precision copy starts as the rounded master
        if w.stage < 3 and w.rank >= 0:
            S = w.shard
            self.params[w.rank * S:(w.rank + 1) * S] = self.master.to(self.params.dtype)
        else:
            self.params.copy_(self.master.to(self.params.dtype))

    def group_ranges(self):
        """(first unit, unit count) of each group of a grouped stage-3 workload."""
        out, first = [], 0
        for n in self.w.groups or []:
            out.append((first, n))
            first += n
        return out

    def _alloc_grads(self):
        w = self.w
        dt = TORCH_DTYPE[w.grad_dtype]
        units = self._units()
        lens = [nu if w.rank < 0 else Su for u, nu, Su, off in units]
        self.grads = []   # per unit: list of world tensors
        self.group_grads = None
        if w.groups:
            # per group and rank one buffer with the group's units end to end
            # (the layout the group calls take); the units' grads are views
            self.group_grads = []
            for first, n in self.group_ranges():
                tot = sum(lens[first:first + n])
                bufs = [torch.zeros(tot, dtype=dt, device=self.dev) for _ in range(w.world)]
                self.group_grads.append(bufs)
                off = 0
                for u in range(first, first + n):
                    self.grads.append([b[off:off + lens[u]] for b in bufs])
                    off += lens[u]
            return
        for n in lens:
            self.grads.append([torch.zeros(n, dtype=dt, device=self.dev) for _ in range(w.world)])

    def fwd_runs(self):
        """The stage-3 forward's gather calls (units without groups): see
        forward_runs."""
        return forward_runs(self.w, self.fwd_pairs)

    def bwd_chunks(self):
        """The stage-3 backward's chunks of two units, or None: see
        backward_chunks."""
        return backward_chunks(self.w, self.fwd_pairs)

    def gather_run(self, first: int, n: int, stream):
        """Place a forward run: one unit into the unit buffer, or a pair into
        the two unit buffers in one call."""
        if n == 1:
            z.zero3_gather_unit(self.ctx, first, self.shards[first], self.unit_full, stream)
        else:
            z.zero3_gather_group(self.ctx, first, self.shards[first:first + 2],
                                 [self.unit_full, self.unit_full2], stream)

    def _alloc_shards(self):
        """The other ranks' parameter shards (one-rank view with placement,
        and stage 3) and the stage-3 unit buffer."""
        w = self.w
        self.shards = None
        self.unit_full = None
        dt = TORCH_DTYPE[w.param_dtype]
        if w.stage == 3:
            self.shards = []
            Pmax = 0
            for u, nu, Su, off in self._units():
                row = []
                for k in range(w.world):
                    if w.rank < 0:
                        row.append(self.params[off + k * Su: off + (k + 1) * Su])
                    elif k == w.rank:
                        row.append(self.params[off: off + Su])
                    else:
                        t = torch.zeros(Su, dtype=dt, device=self.dev)
                        kk = synth.key(w.seed, KIND_SHARD, 0, k, u)
                        self._fill(t, valid_len(nu, Su, k), w.param_dtype, kk, w.sigma_master,
                                   index0=k * Su)
                        row.append(t)
                self.shards.append(row)
                Pmax = max(Pmax, Su * w.world)
            self.unit_full = torch.zeros(Pmax, dtype=dt, device=self.dev)
            self.unit_full2 = (torch.zeros(Pmax, dtype=dt, device=self.dev)
                               if self.fwd_pairs and not w.groups else None)
            self.group_fulls = None
            if w.groups:
                # one destination per unit of a group, side by side in one buffer
                sizes = [Su * w.world for u, nu, Su, off in self._units()]
                longest = max(sum(sizes[f:f + n]) for f, n in self.group_ranges())
                self.group_full = torch.zeros(longest, dtype=dt, device=self.dev)
                self.group_fulls = []
                for f, n in self.group_ranges():
                    views, off = [], 0
                    for u in range(f, f + n):
                        views.append(self.group_full[off:off + sizes[u]])
                        off += sizes[u]
                    self.group_fulls.append(views)
        elif w.rank >= 0 and w.gather_after:
            S = w.shard
            self.shards = []
            for k in range(w.world):
                if k == w.rank:
                    self.shards.append(None)   # written by the step itself
                    continue
                t = torch.zeros(S, dtype=dt, device=self.dev)
                kk = synth.key(w.seed, KIND_SHARD, 0, k, 0)
                self._fill(t, valid_len(w.numel, S, k), w.param_dtype, kk, w.sigma_master,
                           index0=k * S)
                self.shards.append(t)

    # ------------------------------------------------------------- inputs

    def fill_grads(self, it: int):
        """Draw iteration `it`'s grads of every rank (and unit) on the device."""
        w = self.w
        sigma = grad_sigma(w, self.scale)
        for (u, nu, Su, off), row in zip(self._units(), self.grads):
            for k in range(w.world):
                key = synth.key(w.seed, synth.KIND_GRAD, it, k, u)
                if w.rank < 0:
                    self._fill(row[k], nu, w.grad_dtype, key, sigma)
                else:
                    self._fill(row[k], valid_len(nu, Su, w.rank), w.grad_dtype, key, sigma,
                               index0=w.rank * Su)
        if w.inject and w.inject[0] == it:
            k = w.inject[1]
            e = inject_index(w, it, k)
            S0 = w.unit_shard(0) if w.units else w.shard     # the planted value is in unit 0
            if w.rank < 0:
                self.grads[0][k][e] = float("inf")
            elif w.rank * S0 <= e < (w.rank + 1) * S0:
                self.grads[0][k][e - w.rank * S0] = float("inf")

    # --------------------------------------------------------------- step

    def _hp(self, t: int):
        """The hyperparameters the step calls get.  With a device scalar
        block bound, the real ones go into the block (zero_prepare_step, then
        a copy on the step's stream) and the calls get values that the
        kernels must ignore."""
        w = self.w
        if self.hyper is None:
            return w.lr, w.beta1, w.beta2, w.eps, t
        d, h = self.hyper
        z.zero_prepare_step(self.ctx, h, w.lr, w.beta1, w.beta2, w.eps, t, self.scale)
        with torch.cuda.stream(self.stream):
            d.copy_(h, non_blocking=True)
        return 0.5, 0.25, 0.125, 1.0, 1

    def launch_step(self, grads_override=None):
        """Launch one whole step (no synchronization).  Returns the t used."""
        w = self.w
        t = self.t + 1
        st = self.stream
        hp = self._hp(t)
        if w.stage < 3 and w.bucket:
            self.launch_buckets(hp, grads_override)
            if self.shards is not None:
                z.zero_allgather(self.ctx, self.shards, self.params, w.param_dtype, st)
        elif w.stage < 3:
            g = grads_override if grads_override is not None else self.grads[0]
            z.zero_step(self.ctx, g, *hp, self.scale, st)
            if self.shards is not None:
                z.zero_allgather(self.ctx, self.shards, self.params, w.param_dtype, st)
        else:
            # with two state sets every unit steps in one pass (loss-scaled or
            # not) and zero3_end_step applies the verdict; with one, a
            # loss-scaled step reduces every unit, then applies once
            one_pass = self.shadow is not None or self.scale <= 0
            z.zero3_begin_step_scaled(self.ctx, self.scale)
            if w.groups:
                pieces = self.group_ranges()

                def gather(i):
                    f, n = pieces[i]
                    z.zero3_gather_group(self.ctx, f, self.shards[f:f + n], self.group_fulls[i], st)

                def update(i):
                    f, n = pieces[i]
                    if one_pass:
                        z.zero3_step_group(self.ctx, f, n, self.group_grads[i], *hp, st)
                    else:
                        z.zero3_reduce_group(self.ctx, f, n, self.group_grads[i], self.scale, st)
            else:
                pieces = [(u, 1) for u in range(len(w.units))]

                def gather(i):
                    z.zero3_gather_unit(self.ctx, i, self.shards[i], self.unit_full, st)

                def update(i):
                    if one_pass:
                        z.zero3_step_unit(self.ctx, i, self.grads[i], *hp, st)
                    else:
                        z.zero3_reduce_unit(self.ctx, i, self.grads[i], self.scale, st)
            if w.groups:                                 # forward
                for i in range(len(pieces)):
                    gather(i)
            else:
                for f, n in self.fwd_runs():
                    self.gather_run(f, n, st)
            chunks = self.bwd_chunks() if one_pass and self.visits == "fused" else None
            if chunks:
                # backward in chunks of two: gather the first, then step
                # each and gather the next in one call
                self.gather_run(chunks[0][0], chunks[0][1], st)
                for c, (f, n) in enumerate(chunks):
                    gf, gn = chunks[c + 1] if c + 1 < len(chunks) else (0, 0)
                    z.zero3_step_units_gather(
                        self.ctx, f, [self.grads[u] for u in range(f, f + n)], *hp, gf,
                        [self.shards[u] for u in range(gf, gf + gn)],
                        [self.unit_full, self.unit_full2][:gn], st)
            elif one_pass and not w.groups and self.visits == "fused" and pieces:
                # backward: after unit i's backward, its update and the
                # gather of unit i-1 in one call
                U = len(pieces)
                gather(U - 1)
                for i in reversed(range(1, U)):
                    z.zero3_step_unit_gather(self.ctx, i, self.grads[i], *hp, i - 1,
                                             self.shards[i - 1], self.unit_full, st)
                update(0)
            else:
                for i in reversed(range(len(pieces))):   # backward
                    gather(i)
                    update(i)
            if self.shadow is not None:
                z.zero3_end_step(self.ctx, st)
            elif self.scale > 0:
                z.zero_step_apply(self.ctx, *hp, st)
        return t

    def bucket_ranges(self):
        w = self.w
        n = w.shard * (w.world if w.rank < 0 else 1)
        return [(off, min(w.bucket, n - off)) for off in range(0, n, w.bucket)]

    def bucket_grads(self, off, cnt, grads=None):
        """Rank k's grads for elements [off, off+cnt) of this view: views into
        the full local grads (or the given constant-size bucket buffers)."""
        if grads is not None:
            return grads
        return [g[min(off, g.numel()):min(off + cnt, g.numel())] for g in self.grads[0]]

    def launch_buckets(self, hp, bucket_buffers=None):
        """One bucketed step; hp = (lr, beta1, beta2, eps, t) as the calls get them."""
        st = self.stream
        z.zero_bucket_begin(self.ctx, self.scale)
        for off, cnt in self.bucket_ranges():
            z.zero_bucket_step(self.ctx, off, cnt, self.bucket_grads(off, cnt, bucket_buffers),
                               *hp, st)
        z.zero_bucket_end(self.ctx, *hp, st)

    def finish_step(self):
        """Read the verdict (synchronizes), advance t and the loss scale."""
        nonfinite, skipped = z.zero_step_status(self.ctx)
        self.skips.append(skipped)
        if not skipped:
            self.t += 1
        if self.scale > 0:
            self.scale, self.good = z.zero_scale_update(self.scale, skipped, self.good,
                                                         self.w.growth_interval)
        return nonfinite, skipped

    def step(self, it: int, draw: bool = True):
        if draw:
            self.fill_grads(it)
        self.launch_step()
        return self.finish_step()

    def state(self):
        """(master, m, v) of the current state set (synchronizes)."""
        if self.shadow is None or z.zero_current_state(self.ctx) == 0:
            return self.master, self.m, self.v
        return self.shadow

    def close(self):
        self.ctx.close()
