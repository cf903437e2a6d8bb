"""Closed forms of the ZeRO memory and communication accounting -- TEST
INFRASTRUCTURE ONLY (part of the oracle).

Exact rational arithmetic (``fractions.Fraction``) so that comparisons with
printed tables are about the tables' rounding, never about float error.

Sources, cited by page title and section:
  [PD] "论文专题讲解：ZeRO：大模型训练的零冗余状态优化": section "显存账"
       (2+2+K bytes per parameter, K = 12 for mixed-precision Adam), section
       "ZeRO-DP 三阶段" (per-device memory of each stage and its
       communication volume), "Table 1: ZeRO-DP Memory", "Table 2: Maximum
       Model Size", "ZeRO-R" (constant-size fused buffers).
  [ZH] "ZeRO 与 FSDP：切分优化器状态、梯度与参数": section "三个级别" and the
       exercise with its answer (13B on 16 cards), ZeroAdam.state_bytes.
  [GW] "guanweilu.cn article 1460": the 7B / 8-card worked accounting.
"""
from __future__ import annotations

from fractions import Fraction

K_ADAM = 12  # bytes of fp32 master + momentum + variance per parameter [PD]


def model_state_bytes(psi, n, stage: int, k: int = K_ADAM) -> Fraction:
    """Per-device bytes of model states with psi parameters over n data-
    parallel ranks.  stage 0 = plain data parallelism (2+2+K)psi;
    1 = P_os: 4psi + K psi/n; 2 = P_os+g: 2psi + (2+K)psi/n;
    3 = P_os+g+p: (4+K)psi/n  ([PD] "ZeRO-DP 三阶段")."""
    psi, n = Fraction(psi), Fraction(n)
    if stage == 0:
        return (4 + k) * psi
    if stage == 1:
        return 4 * psi + k * psi / n
    if stage == 2:
        return 2 * psi + (2 + k) * psi / n
    if stage == 3:
        return (4 + k) * psi / n
    raise ValueError("stage must be 0..3")


def gb(x) -> Fraction:
    """Bytes to GB with GB = 1e9 bytes (the unit Table 1 is printed in)."""
    return Fraction(x) / 10**9


def max_model_size(mp: int, gpus: int, stage: int, mem_bytes=32 * 10**9,
                   k: int = K_ADAM) -> Fraction:
    """Largest psi whose model states fit in mem_bytes per device when mp-way
    model parallelism splits the model and the remaining gpus/mp ranks run
    ZeRO data parallelism ([PD] Table 2, left half).  Each device holds psi/mp
    of the model, so psi_max = mp * M / (bytes per parameter at n = gpus/mp)."""
    nd = Fraction(gpus, mp)
    per_param = model_state_bytes(1, nd, stage, k)
    return Fraction(mp) * Fraction(mem_bytes) / per_param


def comm_elements_per_rank(psi, n, stage: int) -> Fraction:
    """Elements each rank sends per step ([PD] "通信量", [ZH] exercise 2).
    A ring reduce-scatter or all-gather of psi elements ships (n-1)/n * psi
    per rank.  Plain DP all-reduce = reduce-scatter + all-gather; stages 1 and
    2 do exactly those two; stage 3 all-gathers the parameters twice (forward
    and backward) and reduce-scatters the grads once."""
    psi, n = Fraction(psi), Fraction(n)
    one = (n - 1) / n * psi
    if stage in (0, 1, 2):
        return 2 * one
    if stage == 3:
        return 3 * one
    raise ValueError("stage must be 0..3")


def zero_adam_state_bytes(numel: int, world: int) -> int:
    """ZeroAdam.state_bytes(): fp32 master, m and v of one shard of
    ceil(numel / world) elements ([ZH] "从零实现 ZeRO 的 Adam")."""
    shard = -(-numel // world)
    return 3 * shard * 4


def unsharded_adam_state_bytes(numel: int) -> int:
    """The same three fp32 tensors over the whole vector ([ZH] zero_check)."""
    return 3 * numel * 4


def fused_fp32_buffer_bytes(psi) -> Fraction:
    """A fused fp32 buffer over all psi parameters ([PD] "ZeRO-R", C_B)."""
    return 4 * Fraction(psi)


def printed_matches(printed: str, exact: Fraction) -> bool:
    """Does a printed decimal stand for `exact`?  Either rounding or
    truncation to the printed number of decimals is accepted: the tables
    mix the two (e.g. 41.25 -> "41.3", 2218.75 -> "2218")."""
    dec = len(printed.split(".")[1]) if "." in printed else 0
    val = Fraction(printed)
    return abs(val - exact) < Fraction(1, 10**dec)
