"""Benchmark of the ZeRO sharded optimizer step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--extra-workloads A,B|none] [--impl ours|reference]
                    [--no-e2e] [--no-cpu-baseline] [--graph]

One "step" is one pass of the whole hot path over one batch of synthetic
grads already resident in HBM.  For the default workload (GPT-2 XL shape,
1,557,611,200 params, 16 data-parallel ranks on this GPU, fp16 grads and
params, loss scale 2^16) that is one kernel that reduce-scatters (sums the
ranks' grads in rank order), averages, unscales, checks for overflow, runs
Adam on the fp32 state and casts into the full fp16 parameter buffer, reading
the current state set and writing the other; a finalize kernel that makes
the written set current unless the step overflowed; and the read of the
overflow verdict with the loss-scale update.

Prints ONE JSON line (rank 0).  `value` is params updated per second over
all GPUs: K steps between one pair of CUDA events, inputs resident, nothing
between the launches.  A second pass of K steps puts an event pair around
every launch for the per-kernel durations behind `roofline`: the dominant
kernel's algorithmic bytes per launch over its average duration, against the
measured HBM copy bandwidth.  `e2e` repeats the measurement with the grads
copied from pinned host memory every step, the step's result (the updated
parameters) copied back to pinned host memory and the verdict read back;
`cpu_baseline` times the CPU oracle on a bounded sample (all host cores, and
one).  `--graph` also times replays of one step captured in a CUDA graph.

`config` describes what runs and nothing measured (the reference arm prints
the same dictionary); the measurements are in `measured`, `roofline`, `e2e`
and, for the default run, `workloads`: the 7.5B one-rank view with its
placement, GPT-2 small and the two ZeRO-3 unit paths, each timed after the
headline in a runner of its own (with its own clocks and e2e).

With --gpus N > 1 (torchrun), the workload's W data-parallel ranks (16 for
the headline; --dp-ranks W to choose) are spread over the N processes, W/N
consecutive ranks each, every process one library view of its ranks,
stepped through the library's sharded step (per held rank an all-to-all of
its grad pieces, the process's one fused pass over its shards, a MAX
all-reduce of the flag word, the finalize and an all-gather of the cast
shards; NCCL, or gloo through host memory with --dist-backend gloo).  The
workload is the same at every N: strong scaling, and with N = 1 (--sharded:
a group of one, no collective) it is the headline's step.  --replicas instead runs one full
replica of the workload per GPU with no data-path collective (weak
scaling).
`--impl reference` times the CPU oracle instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

# DRAM bytes (read + write) per launch of the dominant kernel and the ncu
# duration of that launch in us (cold and serialized), from one-pass ncu
# captures of dram__bytes_read.sum + dram__bytes_write.sum and
# gpu__time_duration.sum on cases of a few GB (summarised under profiles/),
# scaled to a full launch by the elements it processes where the case is
# smaller (reads grow in proportion; the few tens of MB of writes still in
# L2 when a launch ends do not, so a scaled write figure is slightly low).
# Each entry is valid only for the kernel source it was taken on (sha256
# prefix); otherwise bench reports null.
TRAFFIC = {
    # 60,000,000-element case (16 fp16 ranks, two state sets), x 25.96
    ("gpt2_xl", "fused_step_kernel"): ("dd04a6e84427b70e", 68.538e9 + 20.968e9, 13178.4),
    # 63 shards of 10,000,000 elements, x 11.72
    ("one_rank_7p5b", "gather_kernel"): ("eae13d5b2b7affa8", 14.767e9 + 14.136e9, 4094.4),
    # 2 Llama-7B layers: every gather has the full workload's shape
    ("zero3_llama7b", "gather_rows_kernel"): ("eae13d5b2b7affa8", 404.82e6 + 349.29e6, 113.5),
    # the same gathers (2-byte params, the same shard sizes)
    ("zero3_llama7b_fp16", "gather_rows_kernel"): ("eae13d5b2b7affa8", 404.82e6 + 349.29e6,
                                                   113.5),
    # the 7 two-unit visits of one step, averaged (the launches differ in
    # size as the bytes per launch do); the full workload itself
    ("zero3_gpt2_small", "visit_kernel"): ("dd04a6e84427b70e", 95.855e6 + 18.091e6, 29.73),
}
KERNEL_SRC = os.path.join(ROOT, "zero_sharded_optimizer_step_gb300", "csrc",
                          "zero_step_kernels.cu")
GATHER_SRC = os.path.join(ROOT, "zero_sharded_optimizer_step_gb300", "csrc", "zero_gather.cu")


def src_hash(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="gpt2_xl",
                    choices=["gpt2_xl", "gpt2_small", "one_rank_7p5b", "zero3_llama7b", "tiny",
                             "gpt2_xl_bucketed", "zero3_prefetch", "zero3_gpt2_small",
                             "gpt2_xl_adamw", "fsdp2_llama7b", "fsdp2_llama7b_per_param",
                             "gpt2_small_stage1", "zero3_llama7b_fp16", "fsdp2_prefetch",
                             "zero2_overlap"])
    ap.add_argument("--graph", action="store_true",
                    help="also capture one step in a CUDA graph and time its replays")
    ap.add_argument("--unit-fwd-ms", type=float, default=0.25,
                    help="zero3_prefetch: stand-in forward compute per unit (backward = 2x)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--step-blocks-per-sm", type=int, default=2,
                    help="zero2_overlap, --overlap-steps: step-kernel blocks per SM while "
                         "backward runs")
    ap.add_argument("--overlap-steps", action="store_true",
                    help="zero3_prefetch / fsdp2_prefetch: each unit's reduce + Adam also in "
                         "the background, beside the next unit's backward")
    ap.add_argument("--clocks-csv", default=None,
                    help="keep the nvidia-smi samples taken during the timed region here")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--two-pass", action="store_true",
                    help="loss-scaled workloads: the scratch-based two-pass step instead of the "
                         "single pass over two state sets")
    ap.add_argument("--units", type=int, default=0,
                    help="zero3_llama7b / fsdp2_llama7b(_per_param): use this many Llama-7B "
                         "layers (small cases)")
    ap.add_argument("--numel", type=int, default=0,
                    help="override the workload's parameter count (small profiling cases)")
    ap.add_argument("--replicas", action="store_true",
                    help="with --gpus N > 1: N independent replicas of the workload (the "
                         "simulated ranks on every GPU) instead of one rank per process")
    ap.add_argument("--dp-ranks", type=int, default=0,
                    help="sharded mode: the data-parallel ranks W spread over the N processes, "
                         "W/N each (default: the workload's own rank count for a flat vector, "
                         "N for stage 3)")
    ap.add_argument("--sharded", action="store_true",
                    help="the sharded mode with one process too (a group of one: the W ranks' "
                         "steps in one process, no collective)")
    ap.add_argument("--dist-backend", default="auto", choices=["auto", "nccl", "gloo"],
                    help="process group backend with --gpus N > 1 (auto: nccl on GPUs); a "
                         "gloo group moves the exchanged data through host memory")
    ap.add_argument("--extra-workloads", default=None,
                    help="comma-separated workloads timed after the headline one ('none': "
                         "only the headline); default: %s for the default run"
                         % ",".join(EXTRA_WORKLOADS))
    return ap.parse_args()


METRIC = "ZeRO step params-updated/s and achieved HBM GB/s vs GB300 peak (1 GPU)"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ------------------------------------------------------------------ clocks

class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, keep=None):
        self.index = index
        self.proc = None
        self.keep = keep        # a path to keep the raw samples at, or None
        self.path = None

    def start(self):
        try:
            if self.keep:
                self.path = self.keep
                os.makedirs(os.path.dirname(os.path.abspath(self.path)), exist_ok=True)
            else:
                fd, self.path = tempfile.mkstemp(prefix="bench_clocks_", suffix=".csv")
                os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index),
                                          "--query-gpu=" + self.Q, "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            if getattr(self, "f", None):
                self.f.close()
            if self.path and not self.keep and os.path.exists(self.path):
                os.unlink(self.path)

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            lines = f.readlines()
        if not self.keep:
            os.unlink(self.path)
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                s, m = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            sm.append(s)
            mx.append(m)
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        loaded = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------- the device timing

class Launch:
    """One kernel launch of the step, bracketed by CUDA events."""

    def __init__(self, name, alg_bytes, fn, kernels=1):
        self.name, self.alg_bytes, self.fn = name, alg_bytes, fn
        self.kernels = kernels      # kernel launches the call makes


class _Library:
    """The binding, imported at the first call through it: a launch plan can
    be built (for its algorithmic bytes) where the library is not loaded."""

    def __getattr__(self, name):
        import zero_sharded_optimizer_step_gb300 as z
        return getattr(z, name)


def step_plan(run):
    """The kernel launches of one step, each with its algorithmic bytes."""
    z = _Library()
    w, st = run.w, run.stream
    bg = 4 if w.grad_dtype == 0 else 2
    bp = 4 if w.param_dtype == 0 else 2
    plan = []
    if w.stage < 3 and w.bucket:
        # constant-size bucket buffers, reused for every bucket of the step
        bufs = run.bucket_buffers
        ranges = run.bucket_ranges()
        n_valid_all = w.numel if w.rank < 0 else min(w.shard, max(0, w.numel - w.rank * w.shard))

        def begin_and(fn):
            return lambda: (z.zero_bucket_begin(run.ctx, run.scale), fn())
        # loss-scaled with one state set: each bucket only reduces into the
        # scratch, and the end applies Adam to every element
        two_pass = run.shadow is None and run.scale > 0
        for i, (off, cnt) in enumerate(ranges):
            nv = max(0, min(cnt, n_valid_all - off))
            fn = (lambda off=off, cnt=cnt: z.zero_bucket_step(
                run.ctx, off, cnt, bufs, w.lr, w.beta1, w.beta2, w.eps, run.t + 1, st))
            if two_pass:
                plan.append(Launch("reduce_kernel", w.world * bg * nv + 4 * cnt,
                                   begin_and(fn) if i == 0 else fn))
            else:
                plan.append(Launch("fused_step_kernel", w.world * bg * nv + (24 + bp) * cnt,
                                   begin_and(fn) if i == 0 else fn))
        n_state = w.shard * (w.world if w.rank < 0 else 1)
        kernels_end = 1 if (run.shadow is not None or run.scale > 0) else 0
        plan.append(Launch("finalize_kernel" if run.shadow is not None else "apply_kernel",
                           (4 + 24 + bp) * n_state if two_pass else 0,
                           lambda: z.zero_bucket_end(run.ctx, w.lr, w.beta1, w.beta2, w.eps,
                                                     run.t + 1, st), kernels=kernels_end))
    elif w.stage < 3:
        n_state = w.shard * (w.world if w.rank < 0 else 1)
        n_valid = w.numel if w.rank < 0 else min(w.shard, max(0, w.numel - w.rank * w.shard))
        if run.shadow is not None:
            # one pass over two state sets; the call also launches the small
            # finalize kernel (flip the current set, or recast on overflow)
            def single():
                z.zero_step(run.ctx, run.grads[0], w.lr, w.beta1, w.beta2, w.eps, run.t + 1,
                            run.scale, st)
            plan.append(Launch("fused_step_kernel", w.world * bg * n_valid + (24 + bp) * n_state,
                               single, kernels=2))
        elif run.scale > 0:
            def red():
                z.zero_step_reduce(run.ctx, run.grads[0], run.scale, st)

            def app():
                z.zero_step_apply(run.ctx, w.lr, w.beta1, w.beta2, w.eps, run.t + 1, st)
            plan.append(Launch("reduce_kernel", w.world * bg * n_valid + 4 * n_state, red))
            plan.append(Launch("apply_kernel", (4 + 24 + bp) * n_state, app))
        else:
            def fused():
                z.zero_step(run.ctx, run.grads[0], w.lr, w.beta1, w.beta2, w.eps, run.t + 1,
                            0.0, st)
            # stage 1 with the all-reduce output also writes the mean grads
            avg = bg * n_state if run.grad_avg is not None else 0
            plan.append(Launch("fused_step_kernel",
                               w.world * bg * n_valid + (24 + bp) * n_state + avg, fused))
        if run.shards is not None:
            n_sh = sum(1 for s in run.shards if s is not None)

            def gat():
                z.zero_allgather(run.ctx, run.shards, run.params, w.param_dtype, st)
            plan.append(Launch("gather_kernel", 2 * bp * w.shard * n_sh, gat))
    else:
        # ZeRO-3: per unit (or per group of units: a layer's parameters, one
        # launch each) a gather before forward, a gather before backward and
        # the unit's update; loss-scaled with two state sets, one pass per
        # unit and zero3_end_step; loss-scaled with one, a reduce per unit and
        # one apply over all units
        shadow = run.shadow is not None
        one_pass = shadow or run.scale <= 0
        if w.groups:
            pieces = run.group_ranges()
        else:
            pieces = [(u, 1) for u in range(len(w.units))]

        def gname(i):
            # the library places a group, or a unit with shards of 32 MiB or
            # more, with gather_rows_kernel; smaller units with gather_kernel
            f, n = pieces[i]
            if w.groups or w.unit_shard(f) * bp >= (32 << 20):
                return "gather_rows_kernel"
            return "gather_kernel"

        def first():
            z.zero3_begin_step_scaled(run.ctx, run.scale)

        def gather(i):
            f, n = pieces[i]
            if w.groups:
                sh = run.shards[f:f + n]
                return lambda: z.zero3_gather_group(run.ctx, f, sh, run.group_fulls[i], st)
            return lambda: z.zero3_gather_unit(run.ctx, f, run.shards[f], run.unit_full, st)

        def update(i):
            f, n = pieces[i]
            if w.groups:
                if one_pass:
                    return lambda: z.zero3_step_group(run.ctx, f, n, run.group_grads[i], w.lr,
                                                      w.beta1, w.beta2, w.eps, run.t + 1, st)
                return lambda: z.zero3_reduce_group(run.ctx, f, n, run.group_grads[i],
                                                    run.scale, st)
            if one_pass:
                return lambda: z.zero3_step_unit(run.ctx, f, run.grads[f], w.lr, w.beta1,
                                                 w.beta2, w.eps, run.t + 1, st)
            return lambda: z.zero3_reduce_unit(run.ctx, f, run.grads[f], run.scale, st)

        def sizes(i):
            f, n = pieces[i]
            S = sum(w.unit_shard(u) for u in range(f, f + n))
            nv = sum(min(w.unit_shard(u), max(0, w.units[u] - w.rank * w.unit_shard(u)))
                     for u in range(f, f + n))
            return S, nv
        def chunk_visit(f, n, gf, gn):
            return lambda: z.zero3_step_units_gather(
                run.ctx, f, [run.grads[u] for u in range(f, f + n)], w.lr, w.beta1, w.beta2,
                w.eps, run.t + 1, gf, [run.shards[u] for u in range(gf, gf + gn)],
                [run.unit_full, run.unit_full2][:gn], st)

        def visit(i):
            # unit i's update and unit i-1's gather in one call
            return lambda: z.zero3_step_unit_gather(run.ctx, i, run.grads[i], w.lr, w.beta1,
                                                    w.beta2, w.eps, run.t + 1, i - 1,
                                                    run.shards[i - 1], run.unit_full, st)
        # the Runner's backward: a unit's update and the next unit's gather as
        # one call, which the library makes one launch when the gathered
        # shards are under 32 MiB (and two, the separate calls', otherwise)
        fused_visits = one_pass and not w.groups and getattr(run, "visits", "fused") == "fused"
        if w.groups:                                             # forward
            for i in range(len(pieces)):
                S, _ = sizes(i)
                plan.append(Launch(gname(i), 2 * bp * S * w.world, gather(i)))
        else:
            # the Runner's forward runs: a unit alone, or a pair in one call
            # (the group gather's row kernel)
            for f, n in run.fwd_runs():
                S = sum(w.unit_shard(u) for u in range(f, f + n))
                plan.append(Launch(gname(f) if n == 1 else "gather_rows_kernel",
                                   2 * bp * S * w.world,
                                   (lambda f=f, n=n: run.gather_run(f, n, st))))
        total_S = 0
        U = len(pieces)
        chunks = run.bwd_chunks() if fused_visits else None
        if chunks:
            # the Runner's backward in chunks of two (one call each: the
            # chunk's steps and the next chunk's gathers)
            def unit_bytes(u):
                # as sizes() counts a unit's step
                S = w.unit_shard(u)
                nv = min(S, max(0, w.units[u] - w.rank * S))
                return w.world * bg * nv + (24 + bp) * S
            f0, n0 = chunks[0]
            S0 = sum(w.unit_shard(u) for u in range(f0, f0 + n0))
            plan.append(Launch(gname(f0) if n0 == 1 else "gather_rows_kernel",
                               2 * bp * S0 * w.world, (lambda f=f0, n=n0: run.gather_run(f, n, st))))
            for c, (f, n) in enumerate(chunks):
                gf, gn = chunks[c + 1] if c + 1 < len(chunks) else (0, 0)
                step_b = sum(unit_bytes(u) for u in range(f, f + n))
                gath_b = 2 * bp * w.world * sum(w.unit_shard(u) for u in range(gf, gf + gn))
                plan.append(Launch("visit_kernel", step_b + gath_b, chunk_visit(f, n, gf, gn)))
                total_S += sum(w.unit_shard(u) for u in range(f, f + n))
        for i in (reversed(range(U)) if not chunks else ()):
            S, nv = sizes(i)
            total_S += S
            step_bytes = w.world * bg * nv + (24 + bp) * S
            if fused_visits:
                if i == U - 1:
                    plan.append(Launch(gname(i), 2 * bp * S * w.world, gather(i)))
                if i == 0:
                    plan.append(Launch("fused_step_kernel", step_bytes, update(i)))
                elif gname(i - 1) == "gather_kernel":
                    Sg, _ = sizes(i - 1)
                    plan.append(Launch("step_gather_kernel", step_bytes + 2 * bp * Sg * w.world,
                                       visit(i)))
                else:
                    Sg, _ = sizes(i - 1)
                    plan.append(Launch("fused_step_kernel", step_bytes, update(i)))
                    plan.append(Launch(gname(i - 1), 2 * bp * Sg * w.world, gather(i - 1)))
                continue
            plan.append(Launch(gname(i), 2 * bp * S * w.world, gather(i)))
            if one_pass:
                plan.append(Launch("fused_step_kernel", step_bytes, update(i)))
            else:
                plan.append(Launch("reduce_kernel", w.world * bg * nv + 4 * S, update(i)))
        if shadow:
            plan.append(Launch("finalize_kernel", 0, lambda: z.zero3_end_step(run.ctx, st)))
        elif run.scale > 0:
            plan.append(Launch("apply_kernel", (4 + 24 + bp) * total_S,
                               lambda: z.zero_step_apply(run.ctx, w.lr, w.beta1, w.beta2,
                                                         w.eps, run.t + 1, st)))
        plan[0] = Launch(plan[0].name, plan[0].alg_bytes,
                         (lambda f=plan[0].fn: (first(), f())))
    return plan


def settle_device_memory():
    """Hand the allocator's cached but unused device blocks back before a
    timed region.  Measured on GB300 (GPT-2 XL step, the same kernel and
    buffers): with about 12 GB of set-up temporaries left cached after the
    grads were allocated the step took 13.45 ms, with them released 13.03."""
    import torch
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def run_step(run, plan, events=None):
    if events is None:
        for L in plan:
            L.fn()
    else:
        for L, (a, b) in zip(plan, events):
            a.record(run.stream)
            L.fn()
            b.record(run.stream)
    if run.scale > 0:
        run.finish_step()          # the verdict decides t and the scale
    else:
        run.t += 1


# Workloads timed after the headline one in the default run, each in its own
# runner (closed before the next): the 7.5B one-rank view with placement, the
# GPT-2 small step and the two ZeRO-3 unit paths.
EXTRA_WORKLOADS = ("one_rank_7p5b", "gpt2_small", "zero3_llama7b", "zero3_gpt2_small")


def make_workload(args, name):
    """The workload `name` with the command line's size overrides; a planted
    overflow is dropped (the timed steps are the ones that apply)."""
    import workloads as W
    sized = ("zero3_llama7b", "fsdp2_llama7b", "fsdp2_llama7b_per_param", "zero3_llama7b_fp16")
    w = W.ALL[name](**({"n_units": args.units} if args.units and name in sized else {}))
    if args.numel and name == args.workload:
        w = w.replace(numel=args.numel, name=w.name + "_numel%d" % args.numel)
    if w.inject:
        w = w.replace(inject=None)
    return w


def uses_shadow(args, w):
    """Loss-scaled workloads step in one pass over two state sets unless
    --two-pass asks for the scratch-based two passes."""
    return w.loss_scale > 0 and not args.two_pass


def path_of(w, shadow):
    return ("single pass over two state sets" if shadow else
            "two passes with an fp32 scratch" if w.loss_scale > 0 else "single pass")


def static_plan_bytes(w, shadow):
    """Algorithmic bytes of one step: the launch plan built on a stand-in for
    the GPU runner (nothing is allocated or launched)."""
    from types import SimpleNamespace

    def bucket_ranges():
        n = w.shard * (w.world if w.rank < 0 else 1)
        return [(off, min(w.bucket, n - off)) for off in range(0, n, w.bucket)]

    def group_ranges():
        out, first = [], 0
        for n in w.groups or []:
            out.append((first, n))
            first += n
        return out
    shards = None
    if w.stage == 3:
        shards = [[None] * w.world for _ in w.units]
    elif w.rank >= 0 and w.gather_after:
        shards = [None if k == w.rank else object() for k in range(w.world)]
    from workloads.runner import backward_chunks, forward_runs
    run = SimpleNamespace(w=w, stream=None, shadow=(None,) if shadow else None,
                          scale=w.loss_scale, grads=[[None]], shards=shards,
                          grad_avg=object() if w.allreduce_out else None, bucket_buffers=None,
                          bucket_ranges=bucket_ranges, group_ranges=group_ranges,
                          group_fulls=[None] * len(w.groups or []), group_grads=None,
                          params=None, unit_full=None, ctx=None, t=0,
                          fwd_runs=lambda: forward_runs(w), gather_run=None,
                          bwd_chunks=lambda: backward_chunks(w))
    return sum(L.alg_bytes for L in step_plan(run))


def workload_config(w, shadow):
    """What a workload is: the same on both arms of the benchmark."""
    return {"workload": describe(w),
            "params_updated_per_step": w.updated_per_step(),
            "alg_bytes_per_step": static_plan_bytes(w, shadow),
            "method_min_bytes_per_param": method_min_bytes(w),
            "bucket_elems": w.bucket or None,
            "path": path_of(w, shadow)}


def extra_names(args):
    if args.extra_workloads is not None:
        return [n for n in args.extra_workloads.split(",") if n and n != "none"]
    default_run = (args.workload == "gpt2_xl" and not args.numel and not args.units
                   and not args.two_pass and not args.graph)
    return list(EXTRA_WORKLOADS) if default_run else []


def static_config(args, world_size):
    """The line's `config`: the headline workload and the others the run
    times, described without any measurement (the reference arm prints the
    same dictionary)."""
    w = make_workload(args, args.workload)
    cfg = workload_config(w, uses_shadow(args, w))
    cfg["l2"] = "inputs larger than L2 (129 MB); no flush between timed steps"
    cfg["parallelism"] = ("%d simulated data-parallel ranks per GPU; %d GPU replica(s)"
                          % (w.world, world_size))
    names = extra_names(args)
    if names:
        cfg["workloads"] = {}
        for n in names:
            x = make_workload(args, n)
            cfg["workloads"][n] = workload_config(x, uses_shadow(args, x))
    return cfg


def measure(args, w, shadow, world_size, device_index, steps, kernel_steps, clocks_csv=None):
    """Time `steps` steps of workload `w` (one pair of CUDA events, nothing
    between the launches), then `kernel_steps` more with an event pair around
    every launch for the per-kernel durations.  Returns (figures, runner,
    plan); the caller closes the runner."""
    import torch

    import workloads as W
    from workloads.runner import Runner

    torch.cuda.set_device(device_index)
    run = Runner(w, device="cuda:%d" % device_index, shadow=shadow, alloc_grads=not w.bucket)
    if w.bucket:
        import synth
        dt = {0: torch.float32, 1: torch.bfloat16, 2: torch.float16}[w.grad_dtype]
        run.bucket_buffers = [torch.empty(w.bucket, dtype=dt, device=run.dev)
                              for _ in range(w.world)]
        for k, b in enumerate(run.bucket_buffers):
            synth.fill_device(b.data_ptr(), w.bucket, w.grad_dtype,
                              synth.key(w.seed, synth.KIND_GRAD, 1, k),
                              W.grad_sigma(w, run.scale), run.stream.cuda_stream)
    else:
        run.fill_grads(1)
    if args.graph:
        # graphs are captured on a stream of their own
        torch.cuda.synchronize()
        run.stream = torch.cuda.Stream(run.dev)
    plan = step_plan(run)
    assert sum(L.alg_bytes for L in plan) == static_plan_bytes(w, shadow)
    settle_device_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(run.stream)
    for _ in range(args.warmup):
        run_step(run, plan)
    e1.record(run.stream)
    torch.cuda.synchronize()
    warm_ms = e0.elapsed_time(e1) / max(1, args.warmup)
    if steps is None:
        # a timed region of at least half a second, for the clock samples
        steps = max(args.steps, min(2000, int(500.0 / max(warm_ms, 1e-3)) + 1))
    if kernel_steps is None:
        kernel_steps = min(steps, max(args.steps, 50))

    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in plan] for _ in range(kernel_steps)]
    clocks = Clocks(device_index, clocks_csv)
    barrier(world_size)
    torch.cuda.synchronize()
    clocks.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(run.stream)
    for _ in range(steps):
        run_step(run, plan)
    t_end.record(run.stream)
    torch.cuda.synchronize()
    barrier(world_size)
    ms = allreduce_max(t_start.elapsed_time(t_end), world_size)
    # the per-kernel durations (the roofline's): events between the launches
    # serialize them, so this pass is not the step time
    torch.cuda.synchronize()
    for k in range(kernel_steps):
        run_step(run, plan, ev[k])
    torch.cuda.synchronize()
    clock_info = clocks.stop()
    barrier(world_size)
    assert all(not s for s in run.skips), "a timed step was skipped"

    per = {}
    for k in range(kernel_steps):
        for L, (a, b) in zip(plan, ev[k]):
            d = per.setdefault(L.name, [0.0, 0])
            d[0] += a.elapsed_time(b)
            d[1] += 1
    dom = max(per, key=lambda n: per[n][0])

    def alg_per_launch(name):
        sel = [L.alg_bytes for L in plan if L.name == name]
        return sum(sel) / len(sel)
    peak, peak_kind = peaks()
    step_ms = ms / steps
    step_bytes = sum(L.alg_bytes for L in plan)
    dom_ms = per[dom][0] / per[dom][1]
    achieved = alg_per_launch(dom) / (dom_ms * 1e-3) / 1e9
    fig = {
        "ms_per_step": step_ms,
        "steps": steps,
        "params_per_s": w.updated_per_step() * world_size / (step_ms * 1e-3),
        "alg_bytes_per_step": step_bytes,
        "step_hbm_gbs": step_bytes / (step_ms * 1e-3) / 1e9,
        "step_frac_of_peak": step_bytes / (step_ms * 1e-3) / 1e9 / peak,
        "peak_gbs": peak,
        "peak_kind": peak_kind,
        "dominant_kernel": {"name": dom, "ms_per_launch": dom_ms,
                            "alg_bytes_per_launch": alg_per_launch(dom),
                            "alg_gbs": achieved, "frac": achieved / peak},
        "per_kernel_ms": {n: per[n][0] / per[n][1] for n in per},
        "per_kernel_alg_gbs": {n: alg_per_launch(n) / (per[n][0] / per[n][1] * 1e-3) / 1e9
                               for n in per if per[n][0] > 0},
        "per_kernel_timing": "%d more steps with an event pair around every launch"
                             % kernel_steps,
        "gpu_launches": sum(L.kernels for L in plan) * steps,
        "working_set_gb": working_set(run) / 1e9,
        "clocks": clock_info,
    }
    return fig, run, plan


def free_memory():
    """Return the device and pinned host memory of a closed runner."""
    import gc

    import torch
    gc.collect()
    torch.cuda.empty_cache()
    if hasattr(torch._C, "_host_emptyCache"):
        torch._C._host_emptyCache()


def bench_ours(args, rank, world_size, device_index):
    w = make_workload(args, args.workload)
    shadow = uses_shadow(args, w)
    fig, run, plan = measure(args, w, shadow, world_size, device_index, args.steps, args.steps,
                             args.clocks_csv)
    dom = fig["dominant_kernel"]
    kh = src_hash(GATHER_SRC if dom["name"] in ("gather_kernel", "gather_rows_kernel")
                  else KERNEL_SRC)
    tr = None if (args.numel or args.units) else TRAFFIC.get((args.workload, dom["name"]))
    traffic = tr[1] if tr and tr[0] == kh else None
    result = {
        "metric": METRIC,
        "value": fig["params_per_s"],
        "unit": "params/s",
        "n_gpus": world_size,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": fig["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "storage": {"grads": "f32 bf16 f16".split()[w.grad_dtype],
                    "params": "f32 bf16 f16".split()[w.param_dtype], "state": "f32"},
        "data": "synthetic (seeded counter-based normal draws; no dataset)",
        "config": static_config(args, world_size),
        "roofline": {
            "kernel": dom["name"],
            "bound": "hbm",
            "achieved": dom["alg_gbs"],
            "peak": fig["peak_gbs"],
            "peak_kind": fig["peak_kind"],
            "unit": "GB/s",
            "frac": dom["frac"],
            "alg_bytes_per_launch": dom["alg_bytes_per_launch"],
            "traffic": traffic,
            # the same ncu capture's duration (cold, serialized) and its DRAM rate
            "traffic_ncu_us": tr[2] if traffic is not None else None,
            "traffic_ncu_gbs": traffic / (tr[2] * 1e3) if traffic is not None else None,
        },
        "measured": {k: fig[k] for k in ("alg_bytes_per_step", "step_hbm_gbs",
                                         "step_frac_of_peak", "per_kernel_ms",
                                         "per_kernel_alg_gbs", "per_kernel_timing",
                                         "working_set_gb")},
        "gpu_launches": fig["gpu_launches"],
        "clocks": fig["clocks"],
    }
    updated = w.updated_per_step()
    if args.graph:
        gms = bench_graph(run, plan, args, world_size)
        result["measured"]["graph_ms_per_step"] = gms
        result["measured"]["graph_params_per_s"] = updated * world_size / (gms * 1e-3)
        result["measured"]["eager_ms_per_step"] = fig["ms_per_step"]
    if not args.no_e2e and not w.bucket:
        result["e2e"] = run_e2e(run, plan, args, world_size)
    if not args.no_cpu_baseline and rank == 0 and world_size == 1:
        result["cpu_baseline"] = cpu_baseline(w, budget_s=12.0)
    run.close()
    del run, plan
    free_memory()
    names = extra_names(args)
    if names:
        result["workloads"] = {}
    for n in names:
        x = make_workload(args, n)
        fx, rx, px = measure(args, x, uses_shadow(args, x), world_size, device_index, None, None)
        if not args.no_e2e and not x.bucket:
            fx["e2e"] = run_e2e(rx, px, args, world_size)
        rx.close()
        del rx, px
        free_memory()
        result["workloads"][n] = fx
    return result


def run_e2e(run, plan, args, world_size):
    w = run.w
    e2e = (bench_e2e_pipelined(run, args, world_size) if w.stage < 3 else
           bench_e2e_units(run, args, world_size) if w.rank >= 0 else None)
    return e2e or bench_e2e(run, plan, args, world_size)


def sharded_workload(args, world_size, rank=0):
    """The workload of the sharded mode: the command line's over W
    data-parallel ranks (--dp-ranks; by default the workload's own rank
    count, or one rank per process when N does not divide it), each of the
    N processes holding W / N consecutive ranks; `rank` is the process's
    index."""
    base = make_workload(args, args.workload)
    # a flat workload must be the all-ranks one (the mode picks each
    # process's ranks); stage-3 workloads are described as one rank's view
    if (base.stage < 3 and base.rank >= 0) or base.bucket or base.groups or base.unit_rows:
        raise SystemExit("the sharded mode steps a flat vector or flat stage-3 units; "
                         "--workload %s is not one (use --replicas)" % args.workload)
    # the workload's own rank count when the processes divide it, else one
    # rank per process (--dp-ranks chooses explicitly)
    W = args.dp_ranks or (base.world if base.world % world_size == 0 else world_size)
    if W % world_size:
        raise SystemExit("--dp-ranks %d is not a multiple of the %d processes" % (W, world_size))
    return base.replace(world=W, rank=rank, name=base.name + "_sharded")


def sharded_config(args, world_size):
    """The sharded mode's `config` (no measurement in it; the reference arm
    prints the same dictionary under the same launch)."""
    w = sharded_workload(args, world_size)
    shards = ([w.shard] if w.stage < 3 else
              [w.unit_shard(u) for u in range(len(w.units))])
    return {
        "workload": describe(w.replace(rank=-1)),
        "params_updated_per_step": sum(shards) * w.world,
        "l2": "inputs larger than L2 (129 MB); no flush between timed steps",
        "parallelism": "%d data-parallel ranks over %d process(es), %d each (one library "
                       "view per process; %s)"
                       % (w.world, world_size, w.world // world_size,
                          ("no collective: a group of one%s"
                           % ("; the unit gathers by the library" if w.stage == 3 else ""))
                          if world_size == 1 else
                          "%s all-to-all of grad slices, MAX all-reduce of the flag word, "
                          "all-gather of the cast shards%s"
                          % (args.dist_backend,
                             ", per unit before forward and backward" if w.stage == 3 else "")),
        "path": path_of(w, w.loss_scale > 0),
    }


def bench_sharded(args, rank, world_size, device_index):
    """The sharded mode (the default for --gpus N > 1; --sharded with one
    process): the workload's W data-parallel ranks over the N processes,
    process p holding ranks p*k .. p*k + k - 1 (k = W/N) in one library
    view of those ranks, stepped through the library's sharded step
    (zero_sharded_optimizer_step_gb300.sharded).  A flat vector (RanksStep):
    per held rank an all-to-all of its grad pieces, the process's one fused
    pass over its k shards, a MAX all-reduce of the flag word, the finalize,
    an all-gather of the cast shards -- with N = 1 no collective, and the
    pass is the headline's single all-ranks launch.  Stage 3 (one rank per
    process): per unit an all-gather before forward and backward and, after
    the unit's backward, the exchange of its grads and its local pass; the
    flag combined after the last unit.  The total work is the whole workload
    whatever N is: strong scaling.  `value` is the elements of all shards
    updated per second."""
    import torch

    import synth
    import workloads as W
    import zero_sharded_optimizer_step_gb300 as z
    from zero_sharded_optimizer_step_gb300 import sharded as sh

    w = sharded_workload(args, world_size, rank)
    torch.cuda.set_device(device_index)
    dev = torch.device("cuda:%d" % device_index)
    st = torch.cuda.current_stream(dev).cuda_stream
    scale = w.loss_scale
    sigma = W.grad_sigma(w, scale)
    bg = 4 if w.grad_dtype == 0 else 2
    bp = 4 if w.param_dtype == 0 else 2
    k = w.world // world_size                  # ranks held by this process
    if w.stage < 3:
        # process `rank` holds ranks rank*k .. rank*k + k - 1 in one view:
        # its k shards end to end, one pass over them
        local = sh.LibraryRank(w.numel, w.world, rank * k, w.grad_dtype, w.param_dtype, dev,
                               shadow=scale > 0, weight_decay=w.weight_decay, n_ranks=k)
        units = [(w.numel, local.shard * k, local.master)]
    else:
        # per unit the process's k shards end to end
        local = sh.LibraryRank3(w.units, w.world, rank * k, w.grad_dtype, w.param_dtype, dev,
                                shadow=scale > 0, weight_decay=w.weight_decay, n_ranks=k)
        units = [(nu, S * k, local.master[o:o + S * k])
                 for nu, S, o in zip(w.units, local.shards, local.offsets)]
    grads, kbytes, updated = [], 0, 0
    for u, (nu, n, master) in enumerate(units):
        # n: the view's range ([rank*n, rank*n + n): k shards, or the unit's shard)
        nv = max(0, min(n, nu - rank * n))
        if nv:
            synth.fill_device(master.data_ptr(), nv, synth.F32,
                              synth.key(w.seed, synth.KIND_MASTER, 0, 0, u), w.sigma_master, st,
                              index0=rank * n)
        for c in range(k):
            g = local.grad_buffer(n * world_size)
            synth.fill_device(g.data_ptr(), nu, w.grad_dtype,
                              synth.key(w.seed, synth.KIND_GRAD, 1, rank * k + c, u), sigma, st)
            grads.append(g)
        kbytes += w.world * bg * nv + (24 + bp) * n
        updated += n * world_size
    if w.stage < 3:
        local.set_master()                     # the params: the filled master's cast
        step = sh.RanksStep(local)
    else:
        for u in range(len(units)):
            local.set_master(u)
        # the next unit's all-gather in flight while a unit is worked on
        step = sh.ShardedZero3Step(local, prefetch=True)
    t, good = 0, 0

    def one():
        nonlocal t, scale, good
        if w.stage < 3:
            _, skipped = step.step(grads, w.lr, w.beta1, w.beta2, w.eps, t + 1,
                                   loss_scale=scale)
        else:
            _, skipped = step.step(lambda u, params: grads[u * k:(u + 1) * k], w.lr, w.beta1,
                                   w.beta2, w.eps, t + 1, loss_scale=scale)
        if scale > 0:
            scale, good = z.zero_scale_update(scale, skipped, good, w.growth_interval)
        if not skipped:
            t += 1
        return skipped

    settle_device_memory()

    def local_only():
        # the process's own kernels alone: the pass over its range (per
        # unit, for stage 3) from the W ranks' pieces -- the exchanged ones,
        # or the local grads in a group of one
        hp = (w.lr, w.beta1, w.beta2, w.eps, t + 1)
        if w.stage < 3:
            local.local_pass(step.pieces(grads), *hp, scale)
            local.finish(*hp)
            return
        local.begin(scale)
        for u in reversed(range(len(units))):
            local.unit_pass(u, step.pieces(u, grads[u * k:(u + 1) * k]), *hp, scale)
        local.finish(*hp)

    for _ in range(args.warmup):
        one()
    torch.cuda.synchronize()
    clocks = Clocks(device_index, args.clocks_csv)
    barrier(world_size)
    torch.cuda.synchronize()
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    skips = [one() for _ in range(args.steps)]
    e1.record()
    torch.cuda.synchronize()
    barrier(world_size)
    ms = allreduce_max(e0.elapsed_time(e1), world_size) / args.steps
    pairs = []
    for _ in range(args.steps):
        torch.cuda.synchronize()
        barrier(world_size)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        local_only()
        b.record()
        local.status()
        pairs.append((a, b))
        t += 1
    torch.cuda.synchronize()
    clock_info = clocks.stop()
    assert not any(skips), "a timed step was skipped"
    kms = allreduce_max(statistics.median(a.elapsed_time(b) for a, b in pairs), world_size)
    e2e = None
    in_bytes = sum(g.numel() * g.element_size() for g in grads)
    local_ranks = int(os.environ.get("LOCAL_WORLD_SIZE", str(world_size)))
    out_bytes = local.params.numel() * local.params.element_size()
    # pinned host copies of the grads in and of the parameter buffer out, the
    # same budget as the single-process e2e
    if (not args.no_e2e
            and in_bytes + out_bytes < 0.3 * host_ram_available() / max(1, local_ranks)):
        # the same steps with this rank's grads copied in from pinned host
        # memory (unit by unit, inside the backward, for stage 3) and its
        # parameter buffer copied back to pinned host memory after the step
        host = [torch.empty(g.numel(), dtype=g.dtype, pin_memory=True).copy_(g) for g in grads]
        out = torch.empty(local.params.numel(), dtype=local.params.dtype, pin_memory=True)
        dgrads = grads

        def one_e2e():
            nonlocal t, scale, good
            if w.stage < 3:
                for d, h in zip(dgrads, host):
                    d.copy_(h, non_blocking=True)
                _, skipped = step.step(dgrads, w.lr, w.beta1, w.beta2, w.eps, t + 1,
                                       loss_scale=scale)
            else:
                def backward(u, params):
                    mine = range(u * k, (u + 1) * k)
                    return [dgrads[i].copy_(host[i], non_blocking=True) for i in mine]
                _, skipped = step.step(backward, w.lr, w.beta1, w.beta2, w.eps, t + 1,
                                       loss_scale=scale)
            out.copy_(local.params, non_blocking=True)
            if scale > 0:
                scale, good = z.zero_scale_update(scale, skipped, good, w.growth_interval)
            if not skipped:
                t += 1

        one_e2e()
        torch.cuda.synchronize()
        barrier(world_size)
        steps = max(2, args.e2e_steps)
        t0 = time.perf_counter()
        for _ in range(steps):
            one_e2e()
        torch.cuda.synchronize()
        dt = allreduce_max(time.perf_counter() - t0, world_size)
        e2e = {"value": updated * steps / dt, "unit": "params/s", "ms_per_step": dt / steps * 1e3,
               "h2d_bytes_per_step": in_bytes * world_size,
               "d2h_bytes_per_step": (out.numel() * out.element_size() + 8) * world_size,
               "per_rank": "its local grads in, its parameter buffer and the verdict out",
               "path": "copies on each rank's compute stream around the sharded step"}
    peak, peak_kind = peaks()
    achieved = kbytes / (kms * 1e-3) / 1e9
    gathers = (2 * bp * sum(u[1] for u in units) * (world_size - 1)
               * (1 if w.stage < 3 else 2))
    res = {
        "metric": METRIC, "value": updated / (ms * 1e-3), "unit": "params/s",
        "n_gpus": world_size, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "f32",
        "storage": {"grads": "f32 bf16 f16".split()[w.grad_dtype],
                    "params": "f32 bf16 f16".split()[w.param_dtype], "state": "f32"},
        "data": "synthetic (seeded counter-based normal draws; no dataset)",
        "config": sharded_config(args, world_size),
        "measured": {"local_kernels_ms": kms, "local_alg_bytes": kbytes,
                     "placed_bytes_per_rank_per_step": gathers,
                     # what the step spends outside the rank's own kernels
                     # (the collectives and their waits); the Paddle page's
                     # profiling advice flags a collective share above 30%
                     "collective_share_of_step": max(0.0, 1.0 - kms / ms),
                     "collective_share_above_30pct": (1.0 - kms / ms) > 0.30,
                     "timing": "K whole steps between one pair of CUDA events on each rank, "
                               "max over ranks; then the rank's own kernels alone, K times"},
        "roofline": {"kernel": "fused_step_kernel", "bound": "hbm", "achieved": achieved,
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": achieved / peak,
                     "alg_bytes_per_launch": kbytes / len(units),
                     "traffic": None},
        # per step: the pass and the finalize (or the reduce and the apply)
        # when loss-scaled, the fused pass alone otherwise; stage 3: one
        # pass per unit, and the finalize (or the apply) when loss-scaled
        # (the unit gathers are the collective's own)
        "gpu_launches": args.steps * ((1 if w.stage < 3 else len(units))
                                      + (1 if scale > 0 else 0)),
        "clocks": clock_info,
    }
    if e2e is not None:
        res["e2e"] = e2e
    local.close()
    return res


def bench_prefetch(args, rank, world_size, device_index):
    """ZeRO-3 with the next unit's gather prefetched on a second stream while
    a stand-in kernel plays the unit's compute: how much gather time stays
    exposed.  Three schedules over the same workload: compute only (no
    gathers), serial (gather, then compute, one stream), overlapped."""
    import torch

    import workloads as W
    from workloads import standin
    from workloads.runner import Runner
    from workloads.zero3_schedule import Zero3Schedule

    if args.workload == "fsdp2_prefetch":
        w = W.fsdp2_llama7b(args.units or 32).replace(name="fsdp2_prefetch")
    else:
        w = W.zero3_llama7b(args.units or 32).replace(name="zero3_prefetch")
    torch.cuda.set_device(device_index)
    run = Runner(w, device="cuda:%d" % device_index)
    run.fill_grads(1)
    sms = torch.cuda.get_device_properties(device_index).multi_processor_count
    blocks = 2 * sms
    sink = torch.empty(blocks * 128, device=run.dev)
    # calibrate the stand-in's iterations to the requested duration
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    probe = 200_000
    for _ in range(2):
        e0.record(run.stream)
        standin.busy(sink.data_ptr(), blocks, probe, run.stream.cuda_stream)
        e1.record(run.stream)
        torch.cuda.synchronize()
    per_iter = e0.elapsed_time(e1) / probe
    it_f = max(1, int(args.unit_fwd_ms / per_iter))
    times = {}
    bg = args.overlap_steps
    clocks = Clocks(device_index, args.clocks_csv)
    clocks.start()
    for mode in ("standin_only" if bg else "compute_only", "serial", "overlap"):
        sch = Zero3Schedule(run, it_f, 2 * it_f, blocks, mode, overlap_steps=bg,
                            step_blocks_per_sm=args.step_blocks_per_sm)
        for _ in range(args.warmup):
            sch.launch_step()
        torch.cuda.synchronize()
        barrier(world_size)
        e0.record(run.stream)
        for _ in range(args.steps):
            sch.launch_step()
        e1.record(run.stream)
        torch.cuda.synchronize()
        times[mode] = allreduce_max(e0.elapsed_time(e1) / args.steps, world_size)
    clock_info = clocks.stop()
    base = times["standin_only" if bg else "compute_only"]
    exposed = times["overlap"] - base
    gathers = times["serial"] - base     # with bg: the gathers and the unit steps
    updated = w.updated_per_step()
    run.close()
    peak, peak_kind = peaks()
    U = len(w.groups) if w.groups else len(w.units)     # visits per direction
    return {
        "metric": METRIC, "value": updated * world_size / (times["overlap"] * 1e-3),
        "unit": "params/s", "n_gpus": world_size, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": times["overlap"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded draws; a stand-in kernel plays each unit's compute)",
        "config": {
            "workload": describe(w) + " + stand-in compute %.3f ms fwd / %.3f ms bwd per %s"
                        % (args.unit_fwd_ms, 2 * args.unit_fwd_ms,
                           "group" if w.groups else "unit"),
            ("standin_only_ms" if bg else "compute_only_ms"): base,
            "serial_ms": times["serial"], "overlap_ms": times["overlap"],
            ("gathers_and_steps_serial_ms" if bg else "gather_time_serial_ms"): gathers,
            ("exposed_gathers_and_steps_ms" if bg else "exposed_gather_ms"): exposed,
            "hidden_fraction": (1 - exposed / gathers) if gathers > 0 else None,
            "gathers_per_step": 2 * U, "standin_blocks": blocks,
            "unit_steps_in_background": bg,
            "step_blocks_per_sm_in_background": args.step_blocks_per_sm if bg else None,
        },
        "roofline": None,
        "gpu_launches": (2 * U + 2 * U + U) * args.steps,
        "clocks": clock_info,
    }


def calibrate_standin(run, blocks, ms):
    """Iterations of the stand-in kernel that take about `ms` on this GPU."""
    import torch

    from workloads import standin
    sink = torch.empty(blocks * 128, device=run.dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    probe = 200_000
    for _ in range(2):
        e0.record(run.stream)
        standin.busy(sink.data_ptr(), blocks, probe, run.stream.cuda_stream)
        e1.record(run.stream)
        torch.cuda.synchronize()
    return max(1, int(ms / (e0.elapsed_time(e1) / probe)))


def bench_zero2_overlap(args, rank, world_size, device_index):
    """The bucketed ZeRO-2 step (GPT-2 XL, 16 fp16 ranks, loss-scaled, two
    state sets) run during backward: each bucket steps on a second stream
    while a stand-in kernel plays the next bucket's backward.  Three
    schedules over the same workload: compute only (no steps), serial (each
    bucket's step after its backward, one stream), overlapped."""
    import torch

    import workloads as W
    from workloads.runner import Runner
    from workloads.zero2_schedule import Zero2Schedule

    w = W.gpt2_xl_bucketed().replace(name="zero2_overlap")
    if args.numel:
        w = w.replace(numel=args.numel)
    torch.cuda.set_device(device_index)
    run = Runner(w, device="cuda:%d" % device_index, shadow=w.loss_scale > 0)
    run.fill_grads(1)
    sms = torch.cuda.get_device_properties(device_index).multi_processor_count
    blocks = 2 * sms
    it_f = calibrate_standin(run, blocks, args.unit_fwd_ms)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = {}
    clocks = Clocks(device_index, args.clocks_csv)
    clocks.start()
    for mode in ("compute_only", "serial", "overlap"):
        sch = Zero2Schedule(run, it_f, 2 * it_f, blocks, mode, args.step_blocks_per_sm)
        for _ in range(args.warmup):
            sch.launch_step()
            if mode != "compute_only":
                run.finish_step()
        torch.cuda.synchronize()
        barrier(world_size)
        e0.record(run.stream)
        for _ in range(args.steps):
            sch.launch_step()
        e1.record(run.stream)
        torch.cuda.synchronize()
        times[mode] = allreduce_max(e0.elapsed_time(e1) / args.steps, world_size)
    clock_info = clocks.stop()
    exposed = times["overlap"] - times["compute_only"]
    steps_serial = times["serial"] - times["compute_only"]
    updated = w.updated_per_step()
    B = len(run.bucket_ranges())
    run.close()
    return {
        "metric": METRIC, "value": updated * world_size / (times["overlap"] * 1e-3),
        "unit": "params/s", "n_gpus": world_size, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": times["overlap"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded draws; a stand-in kernel plays each bucket's compute)",
        "config": {
            "workload": describe(w) + " + stand-in compute %.3f ms fwd / %.3f ms bwd per bucket"
                        % (args.unit_fwd_ms, 2 * args.unit_fwd_ms),
            "compute_only_ms": times["compute_only"], "serial_ms": times["serial"],
            "overlap_ms": times["overlap"], "step_time_serial_ms": steps_serial,
            "exposed_step_ms": exposed,
            "hidden_fraction": (1 - exposed / steps_serial) if steps_serial > 0 else None,
            "buckets": B, "standin_blocks": blocks,
            "step_blocks_per_sm_overlapped": args.step_blocks_per_sm,
            "timing": "loss-scaled steps timed back to back without reading the verdict "
                      "between them (every step applies: no overflow is planted)",
        },
        "roofline": None,
        "gpu_launches": (2 * B + B + 1) * args.steps,
        "clocks": clock_info,
    }


def bench_graph(run, plan, args, world_size):
    """Replays of one step captured in a CUDA graph.  The per-step scalars
    live in a device block (zero_bind_hyper) refreshed by a memcpy node from
    pinned host memory that zero_prepare_step fills before each replay.  Two
    graphs read two host blocks in turn, and a host block is refilled only
    after the replay that read it has run (an event), so one step is always
    queued ahead of the GPU."""
    import torch
    import zero_sharded_optimizer_step_gb300 as z

    w, st = run.w, run.stream
    if run.scale > 0:
        return bench_graph_advance(run, plan, args, world_size)
    hs = [torch.zeros(z.ZERO_HYPER_BYTES, dtype=torch.uint8, pin_memory=True) for _ in range(2)]
    # the scalars go straight into the context's constant slot (one copy per step)
    z.zero_bind_hyper(run.ctx, z.zero_hyper_slot(run.ctx))

    def body(i):
        z.zero_load_hyper(run.ctx, hs[i], st)
        for L in plan:
            L.fn()

    def prepare(i):
        z.zero_prepare_step(run.ctx, hs[i], w.lr, w.beta1, w.beta2, w.eps, run.t + 1, run.scale)

    torch.cuda.synchronize()
    prepare(0)
    body(0)                                 # one eager step in this mode first
    torch.cuda.synchronize()
    run.t += 1
    graphs = [torch.cuda.CUDAGraph() for _ in range(2)]
    for i in range(2):
        with torch.cuda.graph(graphs[i], stream=st):
            body(i)
    read = [torch.cuda.Event(), torch.cuda.Event()]
    started = [False, False]

    def step(k):
        i = k % 2
        if started[i]:
            read[i].synchronize()           # the replay that read hs[i] has run
        prepare(i)
        with torch.cuda.stream(st):
            graphs[i].replay()
        read[i].record(st)
        started[i] = True
        run.t += 1

    for k in range(args.warmup):
        step(k)
    torch.cuda.synchronize()
    barrier(world_size)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for k in range(args.steps):
        step(k)
    e1.record(st)
    torch.cuda.synchronize()
    ms = allreduce_max(e0.elapsed_time(e1) / args.steps, world_size)
    z.zero_bind_hyper(run.ctx, None)
    return ms


def bench_graph_advance(run, plan, args, world_size):
    """Loss-scaled steps replayed from one CUDA graph of [step, advance]: the
    advance kernel reads each step's verdict and rewrites the device block of
    scalars (t, loss scale, bias corrections) for the next, so the host
    neither prepares a step nor reads a verdict between replays."""
    import torch
    import zero_sharded_optimizer_step_gb300 as z

    w, st = run.w, run.stream
    d = torch.zeros(z.ZERO_HYPER_BYTES, dtype=torch.uint8, device=run.dev)
    h = torch.zeros(z.ZERO_HYPER_BYTES, dtype=torch.uint8, pin_memory=True)
    z.zero_bind_hyper(run.ctx, d)
    T = run.t + args.warmup + args.steps + 4
    tab = np.zeros(2 * T, np.float32)
    z.zero_fill_advance_table(tab.ctypes.data, T, w.beta1, w.beta2)
    dtab = torch.from_numpy(tab).to(run.dev)
    hs = np.zeros(4, np.int64)
    z.zero_advance_state(hs.ctypes.data, run.t + 1, run.scale, w.growth_interval)
    ds = torch.from_numpy(hs).to(run.dev)
    z.zero_bind_advance(run.ctx, dtab, T, ds)
    z.zero_prepare_step(run.ctx, h, w.lr, w.beta1, w.beta2, w.eps, run.t + 1, run.scale)
    d.copy_(h)
    torch.cuda.synchronize()

    def body():
        for L in plan:
            L.fn()
        z.zero_advance_step(run.ctx, st)

    with torch.cuda.stream(st):
        body()                              # one eager step in this mode first
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        body()
    with torch.cuda.stream(st):
        for _ in range(args.warmup):
            g.replay()
    torch.cuda.synchronize()
    barrier(world_size)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(st):
        e0.record(st)
        for _ in range(args.steps):
            g.replay()
        e1.record(st)
    torch.cuda.synchronize()
    ms = allreduce_max(e0.elapsed_time(e1) / args.steps, world_size)
    status = int(np.frombuffer(ds.cpu().numpy()[1].tobytes()[4:], np.int32)[0])
    assert status == 0, "the bias table ran out during the graph replays"
    z.zero_bind_advance(run.ctx, None, 0, None)
    z.zero_bind_hyper(run.ctx, None)
    return ms


def working_set(run):
    tot = 0
    for t in [run.master, run.m, run.v, run.params, run.g, run.unit_full,
              *(run.shadow or ())]:
        if t is not None:
            tot += t.numel() * t.element_size()
    for row in run.grads:
        for t in row:
            tot += t.numel() * t.element_size()
    for t in getattr(run, "bucket_buffers", []):
        tot += t.numel() * t.element_size()
    return tot


def method_min_bytes(w):
    bg = 4 if w.grad_dtype == 0 else 2
    bp = 4 if w.param_dtype == 0 else 2
    return w.world * bg + 24 + bp + (bg if w.allreduce_out else 0)


def describe(w):
    if not w.units:
        units = ""
    elif len(set(w.units)) == 1:
        units = " units=%dx%d" % (len(w.units), w.units[0])
    else:
        units = " units=%d (%d to %d elements)" % (len(w.units), min(w.units), max(w.units))
    if w.unit_rows:
        units += " dim-0 row shards"
    if w.groups:
        units += " in %d groups" % len(w.groups)
    if w.allreduce_out:
        units += " all-reduce output"
    return ("%s: numel=%d world=%d stage=%d grad=%s param=%s rank=%s%s%s%s"
            % (w.name, w.numel, w.world, w.stage, "f32 bf16 f16".split()[w.grad_dtype],
               "f32 bf16 f16".split()[w.param_dtype], "all" if w.rank < 0 else w.rank,
               " loss_scale=%g" % w.loss_scale if w.loss_scale else "",
               " weight_decay=%g" % w.weight_decay if w.weight_decay else "", units))


def host_ram_available():
    try:
        return int(open("/proc/meminfo").read().split("MemAvailable:")[1].split()[0]) * 1024
    except Exception:
        return 32 << 30


def result_view(run):
    """The step's result in device memory, which e2e copies back to the host:
    the full parameter buffer (all ranks), the rank's own shard of it (one
    rank's view), or the rank's persistent parameter shards (stage 3)."""
    w = run.w
    if w.stage < 3 and w.rank >= 0:
        return run.params[w.rank * w.shard:(w.rank + 1) * w.shard]
    return run.params


def bench_e2e(run, plan, args, world_size):
    """Same step, with every rank's grads copied from pinned host memory each
    step, the step's result (result_view) copied back to pinned host memory
    after it, and the verdict word read back to the host."""
    import torch
    import zero_sharded_optimizer_step_gb300 as z

    dev_bufs = [t for row in run.grads for t in row] or list(getattr(run, "bucket_buffers", []))
    h2d = sum(t.numel() * t.element_size() for t in dev_bufs)
    avail = host_ram_available()
    # the ranks on this node share its RAM
    local_ranks = int(os.environ.get("LOCAL_WORLD_SIZE", str(world_size)))
    cap = min(h2d, int(0.3 * avail / max(1, local_ranks)), 64 << 30)
    # pinned host copies of the grads (cycled through when RAM is short)
    host = []
    used = 0
    for t in dev_bufs:
        nb = t.numel() * t.element_size()
        if used + nb > cap and host:
            break
        h = torch.empty(t.numel(), dtype=t.dtype, pin_memory=True)
        h.copy_(t)
        host.append(h)
        used += nb
    out_dev = result_view(run)
    out_host = torch.empty(out_dev.numel(), dtype=out_dev.dtype, pin_memory=True)
    st = run.stream
    steps = max(2, args.e2e_steps)

    def one():
        with torch.cuda.stream(st):
            for i, t in enumerate(dev_bufs):
                t.copy_(host[i % len(host)], non_blocking=True)
        for L in plan:
            L.fn()
        with torch.cuda.stream(st):
            out_host.copy_(out_dev, non_blocking=True)
        z.zero_step_status(run.ctx)       # 8-byte read of the verdict
        if run.scale > 0:
            run.scale, run.good = z.zero_scale_update(run.scale, False, run.good,
                                                      run.w.growth_interval)
        run.t += 1

    one()
    torch.cuda.synchronize()
    barrier(world_size)
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    torch.cuda.synchronize()
    dt = allreduce_max(time.perf_counter() - t0, world_size)
    d2h = out_dev.numel() * out_dev.element_size()
    return {"value": run.w.updated_per_step() * world_size * steps / dt, "unit": "params/s",
            "ms_per_step": dt / steps * 1e3, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h + 8, "d2h_result_bytes": d2h, "d2h_verdict_bytes": 8,
            "host_buffers_distinct": len(host), "device_buffers": len(dev_bufs),
            "path": "whole-step copies on the step's stream"}


class ResultCopy:
    """The device-to-host copy of a step's result on a stream of its own,
    started once the step's last kernel is done, so that it runs while the
    next step's host-to-device copies go the other way over the link.  The
    result is copied in pieces; the next step's first write into piece i
    waits for piece i's copy (wait_before_write)."""

    def __init__(self, run, pieces):
        import torch
        self.torch = torch
        self.dev = result_view(run)
        self.host = torch.empty(self.dev.numel(), dtype=self.dev.dtype, pin_memory=True)
        self.stream = torch.cuda.Stream(run.dev)
        self.pieces = pieces                     # (offset, count) into the result
        self.done = [torch.cuda.Event() for _ in pieces]
        self.issued = False
        self.pairs = []
        self.bytes = self.dev.numel() * self.dev.element_size()

    def wait_before_write(self, stream, i):
        if self.issued:
            stream.wait_event(self.done[i])

    def start(self, after_stream, record=False):
        torch = self.torch
        ready = torch.cuda.Event()
        ready.record(after_stream)
        with torch.cuda.stream(self.stream):
            self.stream.wait_event(ready)
            if record:
                self.pairs.append((torch.cuda.Event(enable_timing=True),
                                   torch.cuda.Event(enable_timing=True)))
                self.pairs[-1][0].record(self.stream)
            for (off, cnt), ev in zip(self.pieces, self.done):
                if cnt > 0:
                    self.host[off:off + cnt].copy_(self.dev[off:off + cnt], non_blocking=True)
                ev.record(self.stream)
            if record:
                self.pairs[-1][1].record(self.stream)
        self.issued = True

    def report(self, steps):
        ms = sum(a.elapsed_time(b) for a, b in self.pairs) / max(1, steps)
        return {"d2h_copy_ms_per_step": ms,
                "d2h_gbs_while_stepping": self.bytes / (ms * 1e-3) / 1e9 if ms > 0 else None}


def bench_e2e_pipelined(run, args, world_size, bucket=1 << 25):
    """The end-to-end step through the bucketed API: while bucket b is
    stepped on the compute stream, bucket b+1's grads of every rank are
    copied from pinned host memory on a copy stream into the other of two
    device buffer sets; once the step's verdict is applied (zero_bucket_end)
    its result -- the full parameter buffer, or the rank's own shard of it --
    goes back to pinned host memory on a third stream, beside the next step's
    host-to-device copies; the verdict word is read back.  Same result as
    zero_step; the host link bounds it."""
    import torch
    import zero_sharded_optimizer_step_gb300 as z

    w = run.w
    srcs = run.grads[0]                       # rank k's local grads (or slices)
    h2d = sum(t.numel() * t.element_size() for t in srcs)
    out = result_view(run)
    avail = host_ram_available()
    local_ranks = int(os.environ.get("LOCAL_WORLD_SIZE", str(world_size)))
    if h2d + out.numel() * out.element_size() > int(0.3 * avail / max(1, local_ranks)):
        return None                           # not enough pinned RAM for distinct inputs
    host = []
    for t in srcs:
        h = torch.empty(t.numel(), dtype=t.dtype, pin_memory=True)
        h.copy_(t)
        host.append(h)
    dev = [[torch.empty(bucket, dtype=srcs[0].dtype, device=run.dev) for _ in srcs]
           for _ in range(2)]
    cp = torch.cuda.Stream(run.dev)
    st = run.stream
    ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    n_range = w.shard * (w.world if w.rank < 0 else 1)
    n_valid = srcs[0].numel()
    ranges = [(off, min(bucket, n_range - off)) for off in range(0, n_range, bucket)]
    # the result in the same pieces as the buckets: bucket b's step writes
    # only piece b, so it waits only for piece b of the previous result
    back = ResultCopy(run, ranges)

    pairs = []        # event pairs around each bucket's copies (timed steps)

    def one(record=False):
        z.zero_bucket_begin(run.ctx, run.scale)
        for b, (off, cnt) in enumerate(ranges):
            k2 = b % 2
            nv = max(0, min(cnt, n_valid - off))
            with torch.cuda.stream(cp):
                if b >= 2:
                    cp.wait_event(done[k2])    # the step of bucket b-2 is done with this set
                if record:
                    pairs.append((torch.cuda.Event(enable_timing=True),
                                  torch.cuda.Event(enable_timing=True)))
                    pairs[-1][0].record(cp)
                for d, h in zip(dev[k2], host):
                    if nv:
                        d[:nv].copy_(h[off:off + nv], non_blocking=True)
                if record:
                    pairs[-1][1].record(cp)
                ready[k2].record(cp)
            st.wait_event(ready[k2])
            back.wait_before_write(st, b)
            z.zero_bucket_step(run.ctx, off, cnt, [d[:max(nv, 1)] for d in dev[k2]], w.lr,
                               w.beta1, w.beta2, w.eps, run.t + 1, st)
            done[k2].record(st)
        z.zero_bucket_end(run.ctx, w.lr, w.beta1, w.beta2, w.eps, run.t + 1, st)
        back.start(st, record)                 # the result, final now, back to the host
        if run.shards is not None:
            z.zero_allgather(run.ctx, run.shards, run.params, w.param_dtype, st)
        nonfinite, skipped = z.zero_step_status(run.ctx)   # 8-byte read of the verdict
        if run.scale > 0:
            run.scale, run.good = z.zero_scale_update(run.scale, skipped, run.good,
                                                      w.growth_interval)
        if not skipped:
            run.t += 1

    one()
    torch.cuda.synchronize()
    barrier(world_size)
    steps = max(2, args.e2e_steps)
    t0 = time.perf_counter()
    for _ in range(steps):
        one(record=True)
    torch.cuda.synchronize()                  # the last result copy included
    dt = allreduce_max(time.perf_counter() - t0, world_size)
    copy_ms = sum(a.elapsed_time(b) for a, b in pairs) / steps
    res = {"value": w.updated_per_step() * world_size * steps / dt, "unit": "params/s",
           "ms_per_step": dt / steps * 1e3, "h2d_bytes_per_step": h2d,
           # the time the copy stream spent copying, and the link rate it saw
           "h2d_copy_ms_per_step": copy_ms,
           "h2d_gbs_while_stepping": h2d / (copy_ms * 1e-3) / 1e9 if copy_ms > 0 else None,
           "d2h_bytes_per_step": back.bytes + 8, "d2h_result_bytes": back.bytes,
           "d2h_verdict_bytes": 8,
           "d2h_result": ("the full parameter buffer" if w.rank < 0 else
                          "rank %d's own shard of the parameter buffer" % w.rank),
           "host_buffers_distinct": len(host) + 1, "device_buffers": len(srcs)}
    res.update(back.report(steps))
    res["path"] = ("bucketed step (%d-element buckets) overlapped with the host-to-device "
                   "copies of the next bucket; the result's copy back overlaps the next "
                   "step's" % bucket)
    return res


def bench_e2e_units(run, args, world_size):
    """ZeRO-3 end to end: each unit's grads (all ranks' slices; for a grouped
    workload each group's per-rank buffers) are copied from pinned host memory
    on a copy stream into one of two device buffer sets while the previous
    unit is gathered and stepped; after the step the rank's updated parameter
    shards go back to pinned host memory beside the next step's copies; the
    verdict is read back."""
    import torch
    import zero_sharded_optimizer_step_gb300 as z

    w = run.w
    if w.groups:
        pieces = run.group_ranges()
        src = run.group_grads
    else:
        pieces = [(u, 1) for u in range(len(w.units))]
        src = run.grads
    h2d = sum(t.numel() * t.element_size() for row in src for t in row)
    out = result_view(run)
    avail = host_ram_available()
    local_ranks = int(os.environ.get("LOCAL_WORLD_SIZE", str(world_size)))
    if h2d + out.numel() * out.element_size() > int(0.3 * avail / max(1, local_ranks)):
        return None
    host = []
    for row in src:
        hr = []
        for t in row:
            h = torch.empty(t.numel(), dtype=t.dtype, pin_memory=True)
            h.copy_(t)
            hr.append(h)
        host.append(hr)
    # two sets of device buffers, each the size of the largest piece
    longest = max(t.numel() for row in src for t in row)
    gdt = src[0][0].dtype
    dev = [[torch.empty(longest, dtype=gdt, device=run.dev) for _ in src[0]]
           for _ in range(2)]
    cp = torch.cuda.Stream(run.dev)
    st = run.stream
    ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    # the result in one piece per unit (or group): a piece's next write is its
    # own update in the next step's backward
    offs = []
    for f, n in pieces:
        lo = z.zero_ctx_unit_param_offset(run.ctx, f)
        hi = (z.zero_ctx_unit_param_offset(run.ctx, f + n) if f + n < len(w.units)
              else out.numel())
        offs.append((lo, hi - lo))
    back = ResultCopy(run, offs)

    def gather(i):
        f, n = pieces[i]
        if w.groups:
            z.zero3_gather_group(run.ctx, f, run.shards[f:f + n], run.group_fulls[i], st)
        else:
            z.zero3_gather_unit(run.ctx, f, run.shards[f], run.unit_full, st)

    one_pass = run.shadow is not None or run.scale <= 0

    def step(i, views):
        f, n = pieces[i]
        if w.groups and one_pass:
            z.zero3_step_group(run.ctx, f, n, views, w.lr, w.beta1, w.beta2, w.eps, run.t + 1,
                               st)
        elif w.groups:
            z.zero3_reduce_group(run.ctx, f, n, views, run.scale, st)
        elif one_pass:
            z.zero3_step_unit(run.ctx, f, views, w.lr, w.beta1, w.beta2, w.eps, run.t + 1, st)
        else:
            z.zero3_reduce_unit(run.ctx, f, views, run.scale, st)

    pairs = []        # event pairs around each piece's copies (timed steps)

    def one(record=False):
        z.zero3_begin_step_scaled(run.ctx, run.scale)
        if w.groups:                                         # forward gathers
            for i in range(len(pieces)):
                gather(i)
        else:
            for f, n in run.fwd_runs():
                run.gather_run(f, n, st)
        for j, i in enumerate(reversed(range(len(pieces)))):  # backward
            k2 = j % 2
            views = [d[:h.numel()] for d, h in zip(dev[k2], host[i])]
            with torch.cuda.stream(cp):
                if j >= 2:
                    cp.wait_event(done[k2])
                if record:
                    pairs.append((torch.cuda.Event(enable_timing=True),
                                  torch.cuda.Event(enable_timing=True)))
                    pairs[-1][0].record(cp)
                for d, h in zip(views, host[i]):
                    d.copy_(h, non_blocking=True)
                if record:
                    pairs[-1][1].record(cp)
                ready[k2].record(cp)
            gather(i)
            st.wait_event(ready[k2])
            back.wait_before_write(st, i)
            step(i, views)
            done[k2].record(st)
        # the finalize (which recasts every unit on a skipped step) and the
        # apply come after every unit's update, each of which waited for its
        # piece of the previous result
        if run.shadow is not None:
            z.zero3_end_step(run.ctx, st)
        elif run.scale > 0:
            z.zero_step_apply(run.ctx, w.lr, w.beta1, w.beta2, w.eps, run.t + 1, st)
        back.start(st, record)
        _, skipped = z.zero_step_status(run.ctx)             # 8-byte read of the verdict
        if run.scale > 0:
            run.scale, run.good = z.zero_scale_update(run.scale, skipped, run.good,
                                                      w.growth_interval)
        if not skipped:
            run.t += 1

    one()
    torch.cuda.synchronize()
    barrier(world_size)
    steps = max(2, args.e2e_steps)
    t0 = time.perf_counter()
    for _ in range(steps):
        one(record=True)
    torch.cuda.synchronize()
    dt = allreduce_max(time.perf_counter() - t0, world_size)
    copy_ms = sum(a.elapsed_time(b) for a, b in pairs) / steps
    res = {"value": w.updated_per_step() * world_size * steps / dt, "unit": "params/s",
           "ms_per_step": dt / steps * 1e3, "h2d_bytes_per_step": h2d,
           # the time the copy stream spent copying, and the link rate it saw
           "h2d_copy_ms_per_step": copy_ms,
           "h2d_gbs_while_stepping": h2d / (copy_ms * 1e-3) / 1e9 if copy_ms > 0 else None,
           "d2h_bytes_per_step": back.bytes + 8, "d2h_result_bytes": back.bytes,
           "d2h_verdict_bytes": 8,
           "d2h_result": "rank %d's persistent parameter shards of every unit" % w.rank,
           "host_buffers_distinct": sum(len(r) for r in host) + 1,
           "device_buffers": 2 * len(dev[0])}
    res.update(back.report(steps))
    res["path"] = ("per-%s host-to-device copies overlapped with the previous %s's gather "
                   "and step; the result's copy back overlaps the next step's"
                   % (("group", "group") if w.groups else ("unit", "unit")))
    return res


# ---------------------------------------------------------------- the oracle

def oracle_sample(w, n_s):
    """Inputs of a bounded contiguous sample of the workload for the oracle."""
    import synth
    import workloads as W
    grads = [synth.fill_host(n_s, w.grad_dtype, synth.key(w.seed, synth.KIND_GRAD, 1, k),
                             W.grad_sigma(w, w.loss_scale)) for k in range(w.world)]
    x = synth.fill_host(n_s, synth.F32, synth.key(w.seed, synth.KIND_MASTER), w.sigma_master)
    return grads, x


def host_threads():
    """Host cores this process may run on."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except (AttributeError, OSError):
        return max(1, os.cpu_count() or 1)


def oracle_time(w, n_s, steps, threads=1):
    """Wall seconds of each oracle step over a contiguous n_s-element sample,
    split into `threads` contiguous pieces, one thread per piece.  The update
    is elementwise, so the pieces are independent, and the C oracle runs
    without the interpreter lock.  Returns (elements per step, times)."""
    import threading
    import oracle
    grads, x0 = oracle_sample(w, n_s)
    threads = max(1, min(threads, n_s))
    bounds = [(j * n_s // threads, (j + 1) * n_s // threads) for j in range(threads)]
    pieces = []
    for lo, hi in bounds:
        n = hi - lo
        g = [a[lo:hi] for a in grads]
        if w.rank < 0 and w.stage < 3:
            P = oracle.shard_size(n, w.world) * w.world
            x = np.zeros(P, np.float32)
            x[:n] = x0[lo:hi]
            m, v = np.zeros(P, np.float32), np.zeros(P, np.float32)
            out = np.zeros(P, oracle.NP_STORAGE[w.param_dtype])
        else:
            # one rank's view: the piece is part of its shard, rank 0 of world
            x = x0[lo:hi].copy()
            m, v = np.zeros(n, np.float32), np.zeros(n, np.float32)
            out = np.zeros(n, oracle.NP_STORAGE[w.param_dtype])
        pieces.append((n, g, x, m, v, out))

    def step(piece, t):
        n, g, x, m, v, out = piece
        if w.rank < 0 and w.stage < 3:
            oracle.zero_step(g, w.grad_dtype, n, x, m, v, out, w.param_dtype, w.lr, w.beta1,
                             w.beta2, w.eps, t, loss_scale=w.loss_scale,
                             weight_decay=w.weight_decay)
        else:
            oracle.zero_rank_step(g, w.grad_dtype, n * w.world, 0, x, m, v, out,
                                  w.param_dtype, w.lr, w.beta1, w.beta2, w.eps, t,
                                  loss_scale=w.loss_scale, weight_decay=w.weight_decay)

    times = []
    if threads == 1:
        for t in range(1, steps + 1):
            t0 = time.perf_counter()
            step(pieces[0], t)
            times.append(time.perf_counter() - t0)
        return n_s, times
    bar = threading.Barrier(threads + 1)
    errors = []

    def worker(piece):
        try:
            for t in range(1, steps + 1):
                bar.wait()
                step(piece, t)
                bar.wait()
        except Exception as e:        # reported by the main thread
            errors.append(e)
            bar.abort()

    pool = [threading.Thread(target=worker, args=(p,), daemon=True) for p in pieces]
    for th in pool:
        th.start()
    try:
        for t in range(1, steps + 1):
            bar.wait()                    # every thread starts step t
            t0 = time.perf_counter()
            bar.wait()                    # every thread has finished it
            times.append(time.perf_counter() - t0)
    except threading.BrokenBarrierError:
        pass
    for th in pool:
        th.join()
    if errors:
        raise errors[0]
    return n_s, times


def cpu_baseline(w, budget_s=10.0, steps=4):
    """The oracle on the host: one thread, then one thread per core."""
    n_s = 1 << 20
    _, times = oracle_time(w, n_s, 1)
    # scale the sample so that the single-thread steps take about the budget
    n_s = int(min(1 << 26, max(1 << 16, n_s * budget_s / steps / max(times[0], 1e-6))))
    upd, times = oracle_time(w, n_s, steps)
    single = upd / statistics.median(times)
    T = host_threads()
    steps_t = min(32, steps * T)          # the same sample goes T times faster
    upd, times = oracle_time(w, n_s, steps_t, T)
    return {"value": upd / statistics.median(times), "unit": "params/s", "cores": T,
            "kind": "oracle",
            "sample": "contiguous %d-element piece of the workload (%d ranks) split into %d "
                      "contiguous parts, one thread each; %d steps, median step time; C oracle"
                      % (n_s, w.world, T, steps_t),
            "single_thread": {"value": single, "cores": 1,
                              "sample": "the same piece, one thread, %d steps" % steps}}


def bench_reference(args, rank, world_size):
    if rank != 0:
        return None
    w = make_workload(args, args.workload)
    T = host_threads()
    n_s = 1 << 22
    _, warm = oracle_time(w, n_s, max(1, min(args.warmup, 2)), T)
    per = statistics.median(warm)
    # keep the whole run within a few minutes
    n_s = int(max(1 << 16, min(1 << 26, n_s * 3.0 / max(per, 1e-6))))
    _, times = oracle_time(w, n_s, args.steps, T)
    ms = sum(times) * 1e3
    value = n_s * len(times) / (ms * 1e-3)
    cb = {"value": value, "unit": "params/s", "cores": T, "kind": "oracle",
          "sample": "contiguous %d-element piece of %s per step split into %d contiguous parts, "
                    "one thread each; %d timed steps; C oracle" % (n_s, w.name, T, len(times))}
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "params/s",
            "n_gpus": world_size, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms / len(times), "higher_is_better": True,
            "scaling": "strong" if world_size > 1 and not args.replicas else "weak",
            "vs_baseline": None, "dtype": "f32",
            "storage": {"grads": "f32 bf16 f16".split()[w.grad_dtype],
                        "params": "f32 bf16 f16".split()[w.param_dtype], "state": "f32"},
            "data": "synthetic (seeded counter-based normal draws; no dataset)",
            # the very dictionary the GPU arm prints for the same command line
            "config": (sharded_config(args, world_size) if sharded_mode(args, world_size)
                       else static_config(args, world_size)),
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# -------------------------------------------------------------- distributed

def sharded_mode(args, world_size):
    """Whether this command line runs the sharded mode (the default with
    several processes, --sharded with one)."""
    return (world_size > 1 or args.sharded) and not args.replicas


def barrier(world_size):
    if world_size > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(x, world_size):
    if world_size <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main():
    args = parse()
    world_size = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    device = local
    if world_size > 1:
        import torch
        import torch.distributed as dist
        backend = args.dist_backend
        if backend == "auto":
            backend = "nccl" if torch.cuda.is_available() else "gloo"
        args.dist_backend = backend
        if torch.cuda.is_available():
            # one GPU per process; a gloo group may put several on one GPU
            device = local % torch.cuda.device_count()
            torch.cuda.set_device(device)
        dist.init_process_group(backend)
    elif args.sharded and args.impl == "ours":
        # the sharded mode in a group of one
        import torch
        import torch.distributed as dist
        if args.dist_backend == "auto":
            args.dist_backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(args.dist_backend, store=dist.HashStore(), rank=0, world_size=1)
    if args.impl == "reference":
        res = bench_reference(args, rank, world_size)
    else:
        import __graft_entry__
        __graft_entry__.build() if rank == 0 else None
        barrier(world_size)
        if args.workload in ("zero3_prefetch", "fsdp2_prefetch"):
            res = bench_prefetch(args, rank, world_size, device)
        elif args.workload == "zero2_overlap":
            res = bench_zero2_overlap(args, rank, world_size, device)
        elif sharded_mode(args, world_size):
            res = bench_sharded(args, rank, world_size, device)
        else:
            res = bench_ours(args, rank, world_size, device)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if "torch.distributed" in sys.modules:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
