"""Pins of the oracle's layout, reduce-scatter, all-gather and all-reduce by
brute force on tiny sizes and by the identities the pages state.

Layout: "ZeRO 与 FSDP：切分优化器状态、梯度与参数", section 从零实现 ZeRO 的 Adam
(shard = ceil(numel / world), zero-padded tail, rank r owns [r*S, r*S+S)).
Identity: the same page, section 三个级别 (all-reduce = reduce-scatter +
all-gather), and its exercise 2 (each rank sends 2(N-1)/N of the grad size).
"""
import numpy as np
import pytest

import oracle
from oracle import F16, F32, BF16


def test_shard_size_and_owner_brute_force():
    for psi in range(0, 41):
        for n in range(1, 10):
            S = oracle.shard_size(psi, n)
            smallest = next(s for s in range(0, psi + 2) if s * n >= psi)
            assert S == smallest, (psi, n)
            for i in range(S * n):
                r = next(r for r in range(n) if r * S <= i < (r + 1) * S)
                assert oracle.owner(i, psi, n) == r
            assert oracle.owner(S * n, psi, n) == -1
    assert oracle.shard_size(7_500_000_000, 64) == 117_187_500
    assert oracle.shard_size(1_557_611_200, 16) == 97_350_700
    assert oracle.shard_size(19_210, 4) == 4_803
    assert oracle.shard_size(5, 0) == -1


def _int_grads(rng, n, psi, dtype):
    # small integers: every sum below is exact in fp32, so the expected
    # value is plain integer arithmetic
    vals = rng.integers(-50, 51, size=(n, psi)).astype(np.float32)
    if dtype == F32:
        return [v.copy() for v in vals], vals
    return [oracle.cast(v, dtype) for v in vals], vals


@pytest.mark.parametrize("dtype", [F32, BF16, F16])
def test_reduce_scatter_brute_force(dtype):
    rng = np.random.default_rng(1)
    for psi in range(1, 41):
        for n in range(1, 10):
            grads, vals = _int_grads(rng, n, psi, dtype)
            S = oracle.shard_size(psi, n)
            for r in range(n):
                got = oracle.reduce_scatter_sum(grads, dtype, psi, r)
                want = np.zeros(S, np.float64)
                for j in range(S):
                    i = r * S + j
                    if i < psi:
                        want[j] = sum(float(vals[k, i]) for k in range(n))
                np.testing.assert_array_equal(got, want.astype(np.float32))


def test_all_gather_placement_brute_force():
    rng = np.random.default_rng(2)
    for S in range(0, 12):
        for n in range(1, 10):
            shards = [rng.integers(0, 65535, size=S).astype(np.uint16) for _ in range(n)]
            full = oracle.all_gather(shards, BF16)
            assert full.size == n * S
            for r in range(n):
                for j in range(S):
                    assert full[r * S + j] == shards[r][j]


@pytest.mark.parametrize("dtype", [F32, BF16, F16])
def test_reduce_scatter_then_all_gather_is_all_reduce(dtype):
    """RS (then average) on every rank followed by AG == all-reduce mean,
    bit for bit, including the zero padding."""
    rng = np.random.default_rng(3)
    for psi, n in [(19, 4), (33, 8), (7, 9), (64, 1), (3, 5), (1000, 16)]:
        g32 = [rng.normal(0, 1e-2, psi).astype(np.float32) for _ in range(n)]
        grads = g32 if dtype == F32 else [oracle.cast(g, dtype) for g in g32]
        S = oracle.shard_size(psi, n)
        shards = []
        for r in range(n):
            acc = oracle.reduce_scatter_sum(grads, dtype, psi, r)
            g, bad = oracle.average(acc, n)
            assert bad == 0
            shards.append(g)
        gathered = oracle.all_gather(shards, F32)
        ar = oracle.all_reduce_mean(grads, dtype, psi)
        assert gathered.tobytes() == ar.tobytes()
        assert np.all(ar[psi:] == 0) and not np.any(np.signbit(ar[psi:]))
        assert gathered.size == n * S


def test_communication_bytes_counted():
    """Bytes each rank ships in the simulated RS + AG = 2(N-1)/N of the
    padded vector, i.e. the all-reduce volume."""
    rng = np.random.default_rng(4)
    for psi, n in [(19210, 4), (100, 8), (5, 3)]:
        grads = [oracle.cast(rng.normal(0, 1, psi).astype(np.float32), BF16) for _ in range(n)]
        S = oracle.shard_size(psi, n)
        sent = np.zeros(n, np.int64)
        shards = []
        for r in range(n):
            acc = oracle.reduce_scatter_sum(grads, BF16, psi, r, bytes_sent=sent)
            shards.append(oracle.cast(acc, BF16))
        oracle.all_gather(shards, BF16, bytes_sent=sent)
        P = n * S
        for k in range(n):
            assert sent[k] * n == 2 * (n - 1) * P * 2


def test_sum_order_is_rank_order():
    """The sum is taken g_0 + g_1 + ... in rank order: with values where fp32
    addition is not associative, the result is the left-to-right one."""
    a = np.array([1e8], np.float32)
    b = np.array([-1e8], np.float32)
    c = np.array([1.0], np.float32)
    got = oracle.rank_sum([a, b, c], F32, 1, 1)[0]
    assert got == np.float32((np.float32(1e8) + np.float32(-1e8)) + np.float32(1.0)) == 1.0
    got2 = oracle.rank_sum([c, a, b], F32, 1, 1)[0]
    assert got2 == 0.0  # (1 + 1e8) rounds to 1e8, then - 1e8
    # a lone negative zero keeps its sign; padding is +0
    z = np.array([-0.0, 5.0], np.float32)
    out = oracle.rank_sum([z], F32, 2, 1)
    assert np.signbit(out[0]) and out[1] == 0 and not np.signbit(out[1])


def test_single_rank_is_identity():
    rng = np.random.default_rng(5)
    g = rng.normal(0, 1, 37).astype(np.float32)
    acc = oracle.reduce_scatter_sum([g], F32, 37, 0)
    avg, _ = oracle.average(acc, 1)
    assert avg.tobytes() == g.tobytes()
