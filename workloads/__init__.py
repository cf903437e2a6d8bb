"""The synthetic workloads: parameter counts built from the model shapes the
pages' experiments use, and the input recipe (seeded draws from ``synth``).

No arithmetic of the method lives here.

  tiny            MLP Linear(64,256)+GELU+Linear(256,10): 19,210 fp32 params,
                  4 ranks, 3 steps, lr 1e-2 ("ZeRO 与 FSDP…", zero_check).
  gpt2_small      GPT-2 small (d 768, 12 layers, vocab 50257, context 1024):
                  124,439,808 params, 8 ranks, bf16 grads and params, 10 steps.
  gpt2_xl         GPT-2 XL (d 1600, 48 layers; the 1.5B model of "论文专题讲解：
                  ZeRO", Table 5): 1,557,611,200 params, 16 ranks, fp16 grads
                  drawn at N(0,1e-3) times the current loss scale (2^16 at the
                  start), one +inf in rank 5 at iteration 3.
  one_rank_7p5b   rank 0 of 64 for a 7.5B model (the Figure 1 setting of the
                  same page): shard 117,187,500, 64 incoming bf16 slices, then
                  the placement of 64 bf16 shards into the 7.5e9 buffer.
  zero3_llama7b   32 units shaped like a Llama-7B layer (hidden 4096, SwiGLU
                  FFN 11008, no bias): 202,383,360 params each, rank 0 of 8.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Tuple

F32, BF16, F16 = 0, 1, 2
KIND_SHARD = 3   # synthetic parameter shards held by the other ranks


def gpt2_numel(d: int, layers: int, vocab: int = 50257, ctx: int = 1024) -> int:
    per_layer = (2 * 2 * d                 # ln_1, ln_2 (weight, bias)
                 + d * 3 * d + 3 * d       # attn c_attn
                 + d * d + d               # attn c_proj
                 + d * 4 * d + 4 * d       # mlp c_fc
                 + 4 * d * d + d)          # mlp c_proj
    return vocab * d + ctx * d + layers * per_layer + 2 * d


def mlp_numel() -> int:
    return 64 * 256 + 256 + 256 * 10 + 10


def llama_layer_numel(hidden: int = 4096, ffn: int = 11008) -> int:
    return 4 * hidden * hidden + 3 * hidden * ffn + 2 * hidden


@dataclasses.dataclass
class Workload:
    name: str
    numel: int
    world: int
    stage: int
    grad_dtype: int
    param_dtype: int
    rank: int = -1                       # -1: every rank's state on this GPU
    units: Optional[List[int]] = None    # stage 3
    unit_rows: Optional[List[Tuple[int, int]]] = None   # stage 3, dim-0 layout: (rows, row_elems)
    groups: Optional[List[int]] = None   # stage 3: sizes of runs of units stepped as one
    steps: int = 3
    lr: float = 1e-4
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0            # AdamW's decoupled decay; 0 = Adam
    sigma_grad: float = 1e-3
    sigma_master: float = 0.01
    loss_scale: float = 0.0              # initial scale; 0 = off
    growth_interval: int = 2000
    inject: Optional[Tuple[int, int]] = None   # (iteration, rank): one +inf
    gather_after: bool = False           # place the other ranks' shards too
    bucket: int = 0                      # > 0: step bucket by bucket (elements per bucket)
    allreduce_out: bool = False          # stage 1: also write the averaged grads (all-reduce)
    seed: int = 0

    @property
    def shard(self) -> int:
        return -(-self.numel // self.world)

    def unit_shard(self, u: int) -> int:
        if self.unit_rows:
            rows, row = self.unit_rows[u]
            return -(-rows // self.world) * row
        return -(-self.units[u] // self.world)

    def updated_per_step(self) -> int:
        """Owned elements one step updates (the params-updated/s unit)."""
        if self.stage == 3:
            s = sum(self.unit_shard(u) for u in range(len(self.units)))
            return s * (self.world if self.rank < 0 else 1)
        return self.shard * (self.world if self.rank < 0 else 1)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def tiny() -> Workload:
    return Workload("tiny", mlp_numel(), 4, 2, F32, F32, steps=3, lr=1e-2,
                    sigma_grad=0.01, sigma_master=0.01)


def gpt2_small() -> Workload:
    return Workload("gpt2_small", gpt2_numel(768, 12), 8, 2, BF16, BF16, steps=10)


def gpt2_small_stage1() -> Workload:
    """Stage 1 over the GPT-2 small workload, keeping the all-reduced mean
    grads in a full buffer beside the sharded step (ZeRO-1: grads stay whole,
    only the optimizer states are sharded)."""
    return gpt2_small().replace(name="gpt2_small_stage1", stage=1, allreduce_out=True)


def gpt2_xl() -> Workload:
    return Workload("gpt2_xl", gpt2_numel(1600, 48), 16, 2, F16, F16, steps=10,
                    loss_scale=2.0 ** 16, inject=(3, 5))


def one_rank_7p5b(rank: int = 0) -> Workload:
    return Workload("one_rank_7p5b", 7_500_000_000, 64, 2, BF16, BF16, rank=rank, steps=3,
                    gather_after=True)


def zero3_llama7b(n_units: int = 32) -> Workload:
    return Workload("zero3_llama7b", 32 * llama_layer_numel() if n_units == 32
                    else n_units * llama_layer_numel(), 8, 3, BF16, BF16, rank=0,
                    units=[llama_layer_numel()] * n_units, steps=2)


def zero3_llama7b_fp16(n_units: int = 32) -> Workload:
    """The ZeRO-3 Llama-7B-shaped workload in fp16 with loss scaling (2^16):
    every unit's verdict decides the whole step."""
    return zero3_llama7b(n_units).replace(name="zero3_llama7b_fp16", grad_dtype=F16,
                                          param_dtype=F16, loss_scale=2.0 ** 16)


def gpt2_xl_bucketed() -> Workload:
    """GPT-2 XL stepped in 32 Mi-element buckets from constant-size gradient
    buffers (16 ranks x 64 MiB), the way ZeRO-2 reduce-scatters during backward."""
    return gpt2_xl().replace(name="gpt2_xl_bucketed", bucket=1 << 25)


def dim0(shapes, world: int, rank: int = -1, **kw) -> Workload:
    """Stage 3 in FSDP2's per-parameter dim-0 layout; shapes = [(rows, row_elems)]."""
    units = [r * e for r, e in shapes]
    return Workload("dim0", sum(units), world, 3, BF16, BF16, rank=rank, units=units,
                    unit_rows=list(shapes), **kw)


def llama_layer_shapes(hidden: int = 4096, ffn: int = 11008):
    """The parameter tensors of one Llama decoder layer as (rows, row_elems):
    the q, k, v, o projections, gate, up, down, and the two RMSNorm weights."""
    return ([(hidden, hidden)] * 4 + [(ffn, hidden), (ffn, hidden), (hidden, ffn)]
            + [(hidden, 1)] * 2)


def fsdp2_llama7b_per_param(n_units: int = 32) -> Workload:
    """ZeRO-3 over Llama-7B decoder layers in FSDP2's per-parameter dim-0
    layout: one unit per parameter tensor, each sharded by whole rows (rank 0
    of 8), every parameter gathered and stepped on its own.  32 layers hold
    the elements and bytes of zero3_llama7b, in 288 units instead of 32.
    n_units counts layers."""
    return dim0(llama_layer_shapes() * n_units, 8, 0, steps=2).replace(
        name="fsdp2_llama7b_per_param")


def fsdp2_llama7b(n_units: int = 32) -> Workload:
    """The same per-parameter layout with each layer's nine parameters
    gathered and stepped together (one group per layer), as FSDP2 gathers and
    reduces a module's parameters at once."""
    w = fsdp2_llama7b_per_param(n_units)
    return w.replace(name="fsdp2_llama7b", groups=[len(llama_layer_shapes())] * n_units)


def gpt2_xl_adamw() -> Workload:
    """The GPT-2 XL workload with decoupled weight decay 0.1 (AdamW)."""
    return gpt2_xl().replace(name="gpt2_xl_adamw", weight_decay=0.1)


def zero3_gpt2_small() -> Workload:
    """ZeRO-3 over GPT-2 small with one unit per transformer block, plus the
    embeddings and the final norm (rank 0 of 8): 14 small units, where the
    launch overhead of a 42-launch step matters."""
    d, layers, vocab, ctx = 768, 12, 50257, 1024
    block = gpt2_numel(d, 1, vocab=0, ctx=0) - 2 * d
    units = [vocab * d + ctx * d] + [block] * layers + [2 * d]
    return Workload("zero3_gpt2_small", sum(units), 8, 3, BF16, BF16, rank=0, units=units,
                    steps=2)


ALL = {"tiny": tiny, "zero3_gpt2_small": zero3_gpt2_small, "gpt2_xl_bucketed": gpt2_xl_bucketed,
       "gpt2_small": gpt2_small, "gpt2_small_stage1": gpt2_small_stage1,
       "gpt2_xl": gpt2_xl, "gpt2_xl_adamw": gpt2_xl_adamw,
       "one_rank_7p5b": one_rank_7p5b, "zero3_llama7b": zero3_llama7b,
       "zero3_llama7b_fp16": zero3_llama7b_fp16,
       "fsdp2_llama7b": fsdp2_llama7b, "fsdp2_llama7b_per_param": fsdp2_llama7b_per_param}


def grad_sigma(w: Workload, scale: float) -> float:
    """Grads are drawn at sigma_grad times the loss scale in force."""
    return w.sigma_grad * (scale if scale > 0 else 1.0)
