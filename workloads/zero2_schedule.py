"""The bucketed ZeRO-2 step run during backward ("论文专题讲解：ZeRO", section
ZeRO-DP 三阶段, and "ZeRO 与 FSDP…", section 从零实现 ZeRO 的 Adam: the
gradients of a bucket are reduce-scattered as soon as backward has produced
them, while backward goes on with the layers before it).  The model's own
compute is played by a stand-in kernel (workloads/standin.cu) of a set
duration per bucket: forward over the buckets, then backward over them in
reverse order.

Each bucket's step (reduce-scatter + average + Adam + cast, one
zero_bucket_step) may start once backward has produced that bucket's grads.
In the overlapped schedule it runs on a second stream while the stand-in
plays the backward of the next bucket; zero_bucket_end (the verdict of a
loss-scaled step, with two state sets) follows the last bucket, and the next
step's forward waits for it.  A bucket's params may change during backward:
the layers they belong to have had their backward already.
"""
from __future__ import annotations

import torch

import zero_sharded_optimizer_step_gb300 as z

from . import standin


class Zero2Schedule:
    def __init__(self, run, iters_fwd: int, iters_bwd: int, busy_blocks: int,
                 mode: str = "overlap", step_blocks_per_sm: int = 2):
        w = run.w
        assert w.stage < 3 and w.bucket and mode in ("overlap", "serial", "compute_only")
        assert run.scale <= 0 or run.shadow is not None or run.g is not None
        self.run, self.mode = run, mode
        self.iters = {"f": iters_fwd, "b": iters_bwd}
        self.blocks = busy_blocks
        self.sink = torch.empty(busy_blocks * 128, device=run.dev)
        self.ranges = run.bucket_ranges()
        # the steps run in the background; backward gets the higher priority
        self.ss = torch.cuda.Stream(run.dev, priority=0)
        self.cs = torch.cuda.Stream(run.dev, priority=-1)
        self.ready = [torch.cuda.Event() for _ in self.ranges]
        # overlapped, the step kernels leave room on every SM for the
        # backward's blocks (a full-occupancy step holds every register);
        # the last bucket's step, after backward, takes every SM again
        self.cap = step_blocks_per_sm if mode == "overlap" else 0

    def _busy(self, phase, stream):
        standin.busy(self.sink.data_ptr(), self.blocks, self.iters[phase], stream.cuda_stream)

    def launch_step(self):
        """Launch one whole step (no synchronization).  A step without loss
        scaling advances t here; a loss-scaled one leaves t and the scale to
        run.finish_step(), which reads the verdict."""
        run, w = self.run, self.run.w
        overlap = self.mode == "overlap"
        cs = self.cs if overlap else run.stream
        ss = self.ss if overlap else cs
        if cs is not run.stream:
            cs.wait_stream(run.stream)
        hp = (w.lr, w.beta1, w.beta2, w.eps, run.t + 1)
        for _ in self.ranges:                       # forward
            self._busy("f", cs)
        stepping = self.mode != "compute_only"
        if stepping:
            z.zero_bucket_begin(run.ctx, run.scale)
            if overlap:
                ss.wait_stream(cs)                  # nothing of the last step in flight
        for i in reversed(range(len(self.ranges))):  # backward, last bucket first
            self._busy("b", cs)
            if not stepping:
                continue
            off, cnt = self.ranges[i]
            if overlap:
                self.ready[i].record(cs)            # bucket i's grads exist
                ss.wait_event(self.ready[i])
            z.zero_set_step_occupancy(run.ctx, self.cap if i > 0 else 0)
            z.zero_bucket_step(run.ctx, off, cnt, run.bucket_grads(off, cnt), *hp, ss)
        if stepping:
            z.zero_bucket_end(run.ctx, *hp, ss)
        if overlap:
            cs.wait_stream(ss)
            run.stream.wait_stream(cs)
        if run.scale <= 0:
            run.t += 1
