"""ZeroAdam: the optimizer interface of "ZeRO 与 FSDP：切分优化器状态、梯度与参数"
(section 从零实现 ZeRO 的 Adam: ZeroAdam(params, lr, betas, eps) with step(),
zero_grad() and state_bytes()) over the C ABI -- `ZeroAdam` for N
data-parallel ranks simulated on one GPU, `ShardedZeroAdam` with one process
per rank as the page's listing runs it.

Buffer management only.  The model's parameters become views of one flat,
zero-padded parameter buffer (the page's flat vector in parameters() order);
each simulated rank gets a flat gradient buffer with per-parameter views for
its backward to write into; master weights, m and v are fp32 buffers of the
padded length.  step() is one zero_step call: the reduce-scatter, average,
optional unscale and overflow skip, Adam, cast and placement all run in the
library's kernels.
"""
from __future__ import annotations

from typing import Iterable, List

import torch

from . import binding as z

_DT = {torch.float32: z.ZERO_F32, torch.bfloat16: z.ZERO_BF16, torch.float16: z.ZERO_F16}


class ZeroAdam:
    """Sharded mixed-precision Adam (ZeRO stage 2) for `world` ranks on this GPU.

    params        tensors of one dtype (fp32, bf16 or fp16) on one CUDA device;
                  afterwards each is a view of self.flat (same values).
    world         N, the data-parallel ranks simulated here.
    grad_dtype    element type of the ranks' grads (default: the params').
    loss_scale    > 0 turns on loss scaling: grads are divided by it, a step
                  whose grads hold inf/nan is skipped and the scale halved,
                  and it doubles after growth_interval clean steps.  The step
                  runs as one pass over two fp32 state sets.
    weight_decay  decoupled (AdamW) decay; 0 = Adam.
    """

    def __init__(self, params: Iterable[torch.Tensor], world: int, lr: float = 1e-3,
                 betas=(0.9, 0.999), eps: float = 1e-8, weight_decay: float = 0.0,
                 grad_dtype: torch.dtype | None = None, loss_scale: float = 0.0,
                 growth_interval: int = 2000, stream=None):
        self.params: List[torch.Tensor] = list(params)
        if not self.params:
            raise ValueError("ZeroAdam needs at least one parameter")
        dev, pdt = self.params[0].device, self.params[0].dtype
        if dev.type != "cuda" or pdt not in _DT:
            raise ValueError("parameters must be fp32, bf16 or fp16 CUDA tensors")
        for p in self.params:
            if p.device != dev or p.dtype != pdt:
                raise ValueError("all parameters must share one device and dtype")
        gdt = grad_dtype or pdt
        if gdt not in _DT:
            raise ValueError("grad_dtype must be fp32, bf16 or fp16")
        self.lr, (self.beta1, self.beta2), self.eps = lr, betas, eps
        self.world, self.t, self.scale = world, 0, float(loss_scale)
        self.growth_interval, self.good_steps = growth_interval, 0
        self.stream = stream
        self.numel = sum(p.numel() for p in self.params)
        self.ctx = z.zero_init(self.numel, world, 2, _DT[gdt], _DT[pdt], -1)
        P = z.zero_ctx_state_elems(self.ctx)

        # the flat padded parameter vector; parameters become views of it
        self.flat = torch.zeros(P, dtype=pdt, device=dev)
        self._offsets = []
        off = 0
        with torch.no_grad():
            for p in self.params:
                n = p.numel()
                self.flat[off:off + n].copy_(p.reshape(-1))
                p.data = self.flat[off:off + n].view_as(p)
                self._offsets.append((off, n))
                off += n
        f32 = dict(dtype=torch.float32, device=dev)
        self.master = self.flat.float()
        self.m = torch.zeros(P, **f32)
        self.v = torch.zeros(P, **f32)
        self.flag = torch.zeros(1, dtype=torch.int64, device=dev)
        z.zero_bind(self.ctx, self.master, self.m, self.v, self.flat, None, self.flag)
        self._shadow = None
        if self.scale > 0:
            self._shadow = (torch.zeros(P, **f32), torch.zeros(P, **f32), torch.zeros(P, **f32),
                            torch.zeros(1, dtype=torch.int64, device=dev))
            self._shadow[0].copy_(self.master)
            z.zero_bind_shadow(self.ctx, *self._shadow)
        if weight_decay:
            z.zero_set_weight_decay(self.ctx, weight_decay)
        # rank k's flat local gradient (numel elements; the pad needs none)
        self.grads = [torch.zeros(self.numel, dtype=gdt, device=dev) for _ in range(world)]

    def rank_grads(self, rank: int) -> List[torch.Tensor]:
        """Per-parameter views of rank `rank`'s gradient buffer, shaped like
        the parameters (write the rank's backward here)."""
        g = self.grads[rank]
        return [g[off:off + n].view_as(p) for p, (off, n) in zip(self.params, self._offsets)]

    def zero_grad(self) -> None:
        for g in self.grads:
            g.zero_()

    def step(self) -> bool:
        """One optimizer step over the ranks' grads.  Returns True when the
        step was skipped (loss scaling on and a non-finite grad); then t does
        not advance.  With loss scaling the call reads the verdict back (a
        synchronization)."""
        z.zero_step(self.ctx, self.grads, self.lr, self.beta1, self.beta2, self.eps, self.t + 1,
                    self.scale, self.stream)
        if self.scale <= 0:
            self.t += 1
            return False
        _, skipped = z.zero_step_status(self.ctx)
        if not skipped:
            self.t += 1
        self.scale, self.good_steps = z.zero_scale_update(self.scale, skipped, self.good_steps,
                                                          self.growth_interval)
        return skipped

    def state(self):
        """(master, m, v) of the current fp32 state set, padded length."""
        if self._shadow is not None and z.zero_current_state(self.ctx) == 1:
            return self._shadow[:3]
        return self.master, self.m, self.v

    def state_dict(self) -> dict:
        """Copies of the current fp32 state set (master, m, v; every rank's
        shard, padded length), the step count and the loss-scale state.  The
        parameters are the masters cast, restored from them."""
        x, m, v = self.state()
        return {"master": x.clone(), "m": m.clone(), "v": v.clone(), "t": self.t,
                "scale": self.scale, "good_steps": self.good_steps,
                "world": self.world, "numel": self.numel}

    def load_state_dict(self, sd: dict) -> None:
        """Resume from state_dict() of the same model and world, between
        steps (the resume protocol of zero.h at zero_bind: the saved set
        bound, the current-set and flag words cleared)."""
        if (sd["world"], sd["numel"]) != (self.world, self.numel):
            raise ValueError("the state was saved for %d ranks over %d parameters"
                             % (sd["world"], sd["numel"]))
        torch.cuda.synchronize(self.flat.device)
        self.master.copy_(sd["master"])
        self.m.copy_(sd["m"])
        self.v.copy_(sd["v"])
        if self._shadow is not None:
            self._shadow[3].zero_()
        self.flag.zero_()
        self.t, self.scale, self.good_steps = sd["t"], sd["scale"], sd["good_steps"]
        with torch.no_grad():
            self.flat.copy_(self.master)              # a casting copy

    def state_bytes(self) -> int:
        """Bytes of fp32 optimizer state (master, m, v) per rank: 12 * S, as
        the page's ZeroAdam.state_bytes() reports for its shard."""
        return 12 * z.zero_ctx_shard_size(self.ctx, -1)

    def close(self) -> None:
        self.ctx.close()


class ShardedZeroAdam:
    """The pages' ZeroAdam as its listing runs ("ZeRO 与 FSDP…", section 从零
    实现 ZeRO 的 Adam): one process per data-parallel rank, torch.distributed
    initialized, every process holding the whole model and computing its own
    grads.  The parameters become views of one flat, zero-padded buffer of P
    = N*S elements; this rank keeps fp32 master, m and v of its shard only
    (S = ceil(numel / N)).  step() copies the parameters' .grad into one flat
    gradient and runs the sharded step (sharded.ShardedStep over the
    library's one-rank view): the all-to-all of gradient slices, the local
    pass (sum in rank order, average, unscale, Adam, cast), the verdict
    combined over the ranks and the all-gather that leaves every rank's
    parameters updated in place.

    params        tensors of one dtype (fp32, bf16 or fp16) on this process's
                  CUDA device, the same model on every rank; their .grad is
                  this rank's local gradient (None counts as zero).
    loss_scale    > 0 turns on loss scaling (grads divided by it; a step with
                  inf/nan on any rank is skipped on every rank, the scale
                  halved; doubled after growth_interval clean steps), in one
                  pass over two fp32 state sets.
    weight_decay  decoupled (AdamW) decay; 0 = Adam.
    group         the process group (None: the default group).
    bucket_elems  > 0: exchange the gradients bucket by bucket during the
                  backward, as ZeRO-2 does ("ZeRO 与 FSDP…", 从零实现 ZeRO 的
                  Adam, closing note).  The flat vector is cut into buckets of
                  this many elements, last bucket first (backward produces
                  the last parameters' grads first); each parameter's grad is
                  copied into its buckets as soon as it is accumulated and
                  then freed, and a bucket, once complete, is exchanged and
                  stepped at once (in bucket order on every rank).  step()
                  flushes what is left and finishes.  One backward per step
                  (no accumulation over several).  0 (default): step()
                  takes the whole gradient at once.
    """

    def __init__(self, params: Iterable[torch.Tensor], lr: float = 1e-3, betas=(0.9, 0.999),
                 eps: float = 1e-8, weight_decay: float = 0.0, loss_scale: float = 0.0,
                 growth_interval: int = 2000, group=None, bucket_elems: int = 0):
        import torch.distributed as dist

        from .sharded import LibraryRank, ShardedStep
        self.params: List[torch.Tensor] = list(params)
        if not self.params:
            raise ValueError("ShardedZeroAdam needs at least one parameter")
        dev, pdt = self.params[0].device, self.params[0].dtype
        if dev.type != "cuda" or pdt not in _DT:
            raise ValueError("parameters must be fp32, bf16 or fp16 CUDA tensors")
        for p in self.params:
            if p.device != dev or p.dtype != pdt:
                raise ValueError("all parameters must share one device and dtype")
        self.lr, (self.beta1, self.beta2), self.eps = lr, betas, eps
        self.world, self.rank = dist.get_world_size(group), dist.get_rank(group)
        self.t, self.scale = 0, float(loss_scale)
        self.growth_interval, self.good_steps = growth_interval, 0
        self.numel = sum(p.numel() for p in self.params)
        self.local = LibraryRank(self.numel, self.world, self.rank, _DT[pdt], _DT[pdt], dev,
                                 shadow=self.scale > 0, weight_decay=weight_decay)
        flat = self.local.params
        self._offsets = []
        off = 0
        with torch.no_grad():
            for p in self.params:
                n = p.numel()
                flat[off:off + n].copy_(p.reshape(-1))
                p.data = flat[off:off + n].view_as(p)
                self._offsets.append((off, n))
                off += n
        # the own shard's master weights: its params widened (exact)
        self.local.set_master(self.local.own_params.float())
        self._step = ShardedStep(self.local, group)
        self.bucket_elems = int(bucket_elems)
        if self.bucket_elems > 0:
            self._init_buckets(flat.numel())
        else:
            self.flat_grad = self.local.grad_buffer(flat.numel())

    # ---- buckets exchanged during backward

    def _init_buckets(self, P: int) -> None:
        B = self.bucket_elems
        # bucket b covers [lo_b, hi_b), b = 0 the last range of the vector
        self._buckets = []
        hi = P
        while hi > 0:
            lo = max(0, hi - B)
            self._buckets.append((lo, hi))
            hi = lo
        self._hooks = [p.register_post_accumulate_grad_hook(self._grad_ready)
                       for p in self.params]
        self._by_param = {}
        for p, (off, n) in zip(self.params, self._offsets):
            self._by_param[id(p)] = (off, n)
        self._reset_buckets()

    def _reset_buckets(self) -> None:
        self._bufs = {}
        self._next = 0                  # the next bucket to exchange
        self._begun = False
        # elements still awaited per bucket (the padding needs none)
        self._left = [max(0, min(hi, self.numel) - lo) for lo, hi in self._buckets]

    def _buf(self, b: int) -> torch.Tensor:
        if b not in self._bufs:
            lo, hi = self._buckets[b]
            self._bufs[b] = self.local.grad_buffer(hi - lo)
        return self._bufs[b]

    def _grad_ready(self, p: torch.Tensor) -> None:
        off, n = self._by_param[id(p)]
        g = p.grad.reshape(-1)
        with torch.no_grad():
            for b, (lo, hi) in enumerate(self._buckets):
                a, e = max(lo, off), min(hi, off + n)
                if a < e:
                    self._buf(b)[a - lo:e - lo].copy_(g[a - off:e - off])
                    self._left[b] -= e - a
        p.grad = None               # this rank keeps only the buckets in flight
        self._flush(False)

    def _flush(self, all_of_them: bool) -> None:
        """Exchange and step the complete buckets, in bucket order; with
        all_of_them every remaining one (missing grads count as zero)."""
        while self._next < len(self._buckets) and (all_of_them or self._left[self._next] == 0):
            b = self._next
            if not self._begun:
                self._step.begin(self.scale)
                self._begun = True
            lo, hi = self._buckets[b]
            self._step.bucket(lo, self._buf(b), self.lr, self.beta1, self.beta2, self.eps,
                              self.t + 1)
            del self._bufs[b]
            self._next += 1

    def zero_grad(self) -> None:
        for p in self.params:
            p.grad = None

    def step(self) -> bool:
        """One optimizer step over this rank's grads (a collective: every
        rank calls it).  Returns True when the step was skipped on every rank
        (loss scaling on and a non-finite grad on any rank); then t does not
        advance."""
        if self.bucket_elems > 0:
            self._flush(True)
            _, skipped = self._step.end(self.lr, self.beta1, self.beta2, self.eps, self.t + 1)
            self._reset_buckets()
        else:
            with torch.no_grad():
                for p, (off, n) in zip(self.params, self._offsets):
                    dst = self.flat_grad[off:off + n]
                    if p.grad is None:
                        dst.zero_()
                    else:
                        dst.copy_(p.grad.reshape(-1))
            _, skipped = self._step.step(self.flat_grad, self.lr, self.beta1, self.beta2,
                                         self.eps, self.t + 1, loss_scale=self.scale)
        if not skipped:
            self.t += 1
        if self.scale > 0:
            self.scale, self.good_steps = z.zero_scale_update(self.scale, skipped,
                                                              self.good_steps,
                                                              self.growth_interval)
        return skipped

    def state(self):
        """(master, m, v) of this rank's shard, current state set."""
        return self.local.state()

    def state_dict(self) -> dict:
        """This rank's part of a sharded checkpoint ("PaddlePaddle ZeRO优化":
        each rank saves and restores its own shard of the optimizer state):
        copies of its shard's fp32 master, m and v (the current set), the step
        count and the loss-scale state.  The parameters are not included:
        they are the master weights cast, restored from them."""
        x, m, v = self.local.state()
        return {"master": x.clone(), "m": m.clone(), "v": v.clone(), "t": self.t,
                "scale": self.scale, "good_steps": self.good_steps,
                "world": self.world, "rank": self.rank, "numel": self.numel}

    def load_state_dict(self, sd: dict) -> None:
        """Resume from this rank's state_dict() (the same model, world and
        rank), between steps: the saved set becomes the bound set, the
        current-set word and the flag word are cleared, and every rank's
        parameters are cast from the masters and all-gathered -- a
        collective, every rank calls it."""
        from .sharded import gather_params
        if (sd["world"], sd["rank"], sd["numel"]) != (self.world, self.rank, self.numel):
            raise ValueError("the state was saved by rank %d of %d over %d parameters"
                             % (sd["rank"], sd["world"], sd["numel"]))
        loc = self.local
        torch.cuda.synchronize(loc.device)
        loc.master.copy_(sd["master"])
        loc.m.copy_(sd["m"])
        loc.v.copy_(sd["v"])
        if loc.shadow is not None:
            loc.cur.zero_()
        loc.flag.zero_()
        self.t, self.scale, self.good_steps = sd["t"], sd["scale"], sd["good_steps"]
        loc.own_params.copy_(loc.master)              # a casting copy
        gather_params(loc.params, loc.own_params, self._step.group)

    def state_bytes(self) -> int:
        """Bytes of fp32 optimizer state this rank holds: 12 * S, what the
        page's ZeroAdam.state_bytes() reports."""
        return 12 * self.local.shard

    def close(self) -> None:
        for h in getattr(self, "_hooks", []):
            h.remove()
        self.local.close()


# ---- sharded checkpoints across rank counts ("PaddlePaddle ZeRO优化": each
# rank saves and restores its own shard of the optimizer state).  The state
# lives on one flat vector cut into equal shards, so a checkpoint taken over
# N ranks is the vector's first numel elements, whatever N was; these two
# functions move between that whole and the shards of any rank count.  They
# only slice and concatenate (no arithmetic), on whatever device the saved
# tensors are.

_STATE_KEYS = ("master", "m", "v")


def consolidate_state(shards) -> dict:
    """The optimizer state of the whole flat vector from a checkpoint:
    `shards` is either every rank's ShardedZeroAdam.state_dict() (any order,
    ranks 0..N-1 each once) or a single ZeroAdam.state_dict() (which holds
    every rank's shard already).  Returns {"master", "m", "v"} over the
    numel parameters (the padding dropped) with "t", "scale", "good_steps"
    and "numel"; the step count and loss-scale state must agree across
    ranks.  ValueError on an incomplete or inconsistent checkpoint."""
    if isinstance(shards, dict):
        shards = [shards]
    shards = list(shards)
    if not shards:
        raise ValueError("no state to consolidate")
    first = shards[0]
    numel, world = first["numel"], first["world"]
    for sd in shards:
        if (sd["numel"], sd["world"]) != (numel, world):
            raise ValueError("the shards come from different checkpoints")
        if (sd["t"], sd["scale"], sd["good_steps"]) != (first["t"], first["scale"],
                                                        first["good_steps"]):
            raise ValueError("the ranks disagree on the step count or the loss scale")
    if "rank" not in first:                     # ZeroAdam: every shard in one state
        if len(shards) != 1:
            raise ValueError("a ZeroAdam state holds every rank: pass it alone")
        parts = {k: first[k] for k in _STATE_KEYS}
    else:
        by_rank = {sd["rank"]: sd for sd in shards}
        if sorted(by_rank) != list(range(world)) or len(shards) != world:
            raise ValueError("a checkpoint of %d ranks needs each rank's state once (got %s)"
                             % (world, sorted(sd["rank"] for sd in shards)))
        parts = {k: torch.cat([by_rank[r][k].reshape(-1) for r in range(world)])
                 for k in _STATE_KEYS}
    S = z.zero_shard_size(numel, world)
    out = {}
    for k, t in parts.items():
        if t.numel() != S * world:
            raise ValueError("%s holds %d elements, the layout %d" % (k, t.numel(), S * world))
        out[k] = t.reshape(-1)[:numel].clone()
    out.update(t=first["t"], scale=first["scale"], good_steps=first["good_steps"], numel=numel)
    return out


def shard_state(full: dict, world: int, rank: int | None = None) -> dict:
    """The inverse of consolidate_state for `world` ranks: rank `rank`'s
    ShardedZeroAdam.state_dict() (its shard of S = ceil(numel / world)
    elements, zeros past numel), or with rank None a ZeroAdam.state_dict()
    of `world` ranks (every shard, N * S elements).  The result loads with
    load_state_dict into an optimizer of that rank count over the same
    parameters."""
    numel = full["numel"]
    S = z.zero_shard_size(numel, world)
    if S < 0:
        raise ValueError("bad rank count %d" % world)
    lo, n = (0, S * world) if rank is None else (rank * S, S)
    if rank is not None and not 0 <= rank < world:
        raise ValueError("rank %d is not in [0, %d)" % (rank, world))
    out = {}
    for k in _STATE_KEYS:
        src = full[k].reshape(-1)
        part = torch.zeros(n, dtype=src.dtype, device=src.device)
        hi = min(numel, lo + n)
        if hi > lo:
            part[:hi - lo] = src[lo:hi]
        out[k] = part
    out.update(t=full["t"], scale=full["scale"], good_steps=full["good_steps"],
               world=world, numel=numel)
    if rank is not None:
        out["rank"] = rank
    return out

