"""The ZeRO-3 step with the next unit's gather prefetched on a second stream
("ZeRO 与 FSDP：切分优化器状态、梯度与参数", section ZeRO-3 与 FSDP: while
unit i computes, all-gather unit i+1, so the communication hides behind the
computation).  The model's own compute is played by a stand-in kernel
(workloads/standin.cu) of a set duration per unit visit.

Visits: forward over units 0..U-1, then backward over U-1..0, each backward
visit followed by that unit's reduce + Adam.  Two unit buffers alternate:
the gather for visit v+1 writes the buffer visit v-1 used, so it waits for
visit v-1's compute to finish.

With loss scaling the backward visit only reduces (and unscales) its unit's
grads; Adam waits until every unit's overflow flag is in, and one apply pass
after the last visit updates all units or, on overflow, none ("PaddlePaddle
ZeRO优化", section 混合精度才是最佳拍档: the scaler skips the whole step).
With a second state set bound, the backward visit steps its unit in one
pass into that set and zero3_end_step applies the verdict after the last.

A workload with groups of units (FSDP2's per-parameter layout, a layer's
parameters per group) visits groups instead: one group gather and one group
step per visit.
"""
from __future__ import annotations

import torch

import zero_sharded_optimizer_step_gb300 as z

from . import standin


class Zero3Schedule:
    """mode: "overlap" (gathers prefetched in the background), "serial" (all
    on one stream), "compute_only" (no gathers), "standin_only" (neither
    gathers nor steps: the stand-in compute alone).  overlap_steps: in the
    overlap mode, each backward visit's reduce + Adam also runs in the
    background, once the visit's compute is done, beside the next visit's
    compute (the step kernels then take at most step_blocks_per_sm blocks per
    SM, leaving room for the compute's blocks)."""

    def __init__(self, run, iters_fwd: int, iters_bwd: int, busy_blocks: int,
                 mode: str = "overlap", overlap_steps: bool = False, step_blocks_per_sm: int = 2):
        assert run.w.stage == 3 and mode in ("overlap", "serial", "compute_only",
                                             "standin_only")
        self.run, self.mode = run, mode
        self.overlap_steps = overlap_steps and mode == "overlap"
        self.iters = {"f": iters_fwd, "b": iters_bwd}
        self.blocks = busy_blocks
        self.sink = torch.empty(busy_blocks * 128, device=run.dev)
        w = run.w
        # the pieces a visit gathers and steps: single units, or groups of
        # units (a layer's parameters) gathered and stepped in one launch each
        self.pieces = run.group_ranges() if w.groups else [(u, 1) for u in range(len(w.units))]
        if w.groups:
            # two buffers of a group's destinations, alternating between visits
            sizes = [w.unit_shard(u) * w.world for u in range(len(w.units))]
            self.bufs = []
            for big in (run.group_full, torch.empty_like(run.group_full)):
                per_piece = []
                for f, n in self.pieces:
                    views, off = [], 0
                    for u in range(f, f + n):
                        views.append(big[off:off + sizes[u]])
                        off += sizes[u]
                    per_piece.append(views)
                self.bufs.append(per_piece)
        else:
            self.bufs = [run.unit_full, torch.empty_like(run.unit_full)]
        # prefetches run in the background: the lean (bulk-copy) gather leaves
        # the SMs to the compute, which gets the higher stream priority
        self.gs = torch.cuda.Stream(run.dev, priority=0)
        self.cs = torch.cuda.Stream(run.dev, priority=-1)
        self.ss = torch.cuda.Stream(run.dev, priority=0) if self.overlap_steps else None
        # steps beside compute leave room on every SM for its blocks; the
        # last visit's step, after all compute, takes every SM again
        self.cap = step_blocks_per_sm if self.overlap_steps else 0
        z.zero_set_gather_mode(run.ctx, z.ZERO_GATHER_LEAN if mode == "overlap"
                               else z.ZERO_GATHER_FAST)
        U = len(self.pieces)
        self.visits = [(u, "f") for u in range(U)] + [(u, "b") for u in reversed(range(U))]
        n = len(self.visits)
        self.ready = [torch.cuda.Event() for _ in range(n)]
        self.used = [torch.cuda.Event() for _ in range(n)]
        self.grads_done = [torch.cuda.Event() for _ in range(n)]

    def _gather(self, v, stream):
        i, _ = self.visits[v]
        f, n = self.pieces[i]
        run = self.run
        if run.w.groups:
            z.zero3_gather_group(run.ctx, f, run.shards[f:f + n], self.bufs[v % 2][i], stream)
        else:
            z.zero3_gather_unit(run.ctx, f, run.shards[f], self.bufs[v % 2], stream)

    def _compute(self, v, stream):
        i, phase = self.visits[v]
        standin.busy(self.sink.data_ptr(), self.blocks, self.iters[phase], stream.cuda_stream)
        if phase == "b" and self.mode != "standin_only":
            if self.overlap_steps:
                self.grads_done[v].record(stream)   # the unit's backward is done
                self.ss.wait_event(self.grads_done[v])
                stream = self.ss
            z.zero_set_step_occupancy(self.run.ctx, self.cap if v + 1 < len(self.visits) else 0)
            run, w = self.run, self.run.w
            f, n = self.pieces[i]
            two_pass = run.scale > 0 and run.shadow is None
            if w.groups and two_pass:
                z.zero3_reduce_group(run.ctx, f, n, run.group_grads[i], run.scale, stream)
            elif w.groups:
                z.zero3_step_group(run.ctx, f, n, run.group_grads[i], w.lr, w.beta1, w.beta2,
                                   w.eps, run.t + 1, stream)
            elif two_pass:
                z.zero3_reduce_unit(run.ctx, f, run.grads[f], run.scale, stream)
            else:
                z.zero3_step_unit(run.ctx, f, run.grads[f], w.lr, w.beta1, w.beta2,
                                  w.eps, run.t + 1, stream)

    def _apply(self, stream):
        run, w = self.run, self.run.w
        if self.mode == "standin_only":
            return
        if self.overlap_steps:
            stream = self.ss
        if run.shadow is not None:
            z.zero3_end_step(run.ctx, stream)
        elif run.scale > 0:
            z.zero_step_apply(run.ctx, w.lr, w.beta1, w.beta2, w.eps, run.t + 1, stream)

    def launch_step(self):
        """Launch one whole step (no synchronization).  A step without loss
        scaling always applies and advances t here; a loss-scaled one leaves t
        and the scale to run.finish_step(), which reads the verdict."""
        run = self.run
        cs = self.cs if self.mode == "overlap" else run.stream
        if cs is not run.stream:
            cs.wait_stream(run.stream)
        if self.mode != "standin_only":
            z.zero3_begin_step_scaled(run.ctx, run.scale)
        if self.overlap_steps:
            self.ss.wait_stream(cs)                 # nothing of the last step in flight
        n = len(self.visits)
        if self.mode != "overlap":
            for v in range(n):
                if self.mode == "serial":
                    self._gather(v, cs)
                self._compute(v, cs)
            self._apply(cs)
        else:
            gs = self.gs
            gs.wait_stream(cs)            # the shards the last step wrote
            self._gather(0, gs)
            self.ready[0].record(gs)
            for v in range(n):
                cs.wait_event(self.ready[v])
                self._compute(v, cs)
                self.used[v].record(cs)
                if v + 1 < n:
                    if v >= 1:
                        gs.wait_event(self.used[v - 1])   # its buffer is free again
                    self._gather(v + 1, gs)
                    self.ready[v + 1].record(gs)
            self._apply(cs)
            cs.wait_stream(gs)
            if self.overlap_steps:
                cs.wait_stream(self.ss)
            run.stream.wait_stream(cs)
        if run.scale <= 0:
            run.t += 1
