"""Pins of the oracle's type conversions and of the loss-scale skip.

Casts: the fp16/bf16 params are the fp32 master rounded to nearest even
("论文专题讲解：ZeRO", section 显存账: fp16 params next to fp32 master);
checked against numpy's and torch's own conversions.
Skip: "PaddlePaddle ZeRO优化", section 混合精度才是最佳拍档 (GradScaler:
scaler.step skips the update when the unscaled grads hold inf/nan,
scaler.update halves the scale).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import BF16, F16, F32


def _edge_values():
    rng = np.random.default_rng(20)
    vals = [0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, np.nan, 65504.0, 65519.99, 65520.0,
            -65520.0, 6.1e-5, 5.96e-8, 2.98e-8, 2.99e-8, 1e-40, -1e-45,
            3.4028235e38, -3.4028235e38, 3.3961e38, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9,
            1.0 + 2 ** -11, 1.0 + 3 * 2 ** -12]
    bits = rng.integers(0, 2 ** 32, 200000, dtype=np.uint64).astype(np.uint32)
    # ties for bf16: low 16 bits exactly 0x8000
    ties = (rng.integers(0, 2 ** 16, 2000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    ties16 = (rng.integers(0, 2 ** 19, 2000, dtype=np.uint64).astype(np.uint32) << 13) | 0x1000
    x = np.concatenate([np.array(vals, np.float32), bits.view(np.float32),
                        ties.view(np.float32), ties16.view(np.float32),
                        rng.normal(0, 1e-3, 10000).astype(np.float32),
                        (rng.normal(0, 1, 10000) * 65536).astype(np.float32)])
    return x


def test_bf16_cast_matches_torch():
    x = _edge_values()
    got = oracle.cast(x, BF16)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], want[~nan])
    # NaN stays NaN
    assert np.all((got[nan] & 0x7F80) == 0x7F80) and np.all((got[nan] & 0x7F) != 0)


def test_f16_cast_matches_numpy():
    x = _edge_values()
    got = oracle.cast(x, F16)
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.all((got[nan] & 0x7C00) == 0x7C00) and np.all((got[nan] & 0x3FF) != 0)
    # overflow rounds to inf, the largest finite survives
    assert oracle.cast(np.array([65520.0, 65504.0], np.float32), F16).tolist() == [0x7C00, 0x7BFF]


@pytest.mark.parametrize("dtype", [BF16, F16])
def test_widen_is_exact(dtype):
    bits = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.widen(bits, dtype)
    if dtype == F16:
        want = bits.view(np.float16).astype(np.float32)
    else:
        want = (bits.astype(np.uint32) << 16).view(np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))
    # round trip
    assert np.array_equal(oracle.cast(got, dtype)[~nan], bits[~nan])


def test_f32_cast_is_identity():
    x = _edge_values()
    got = oracle.cast(x, F32)
    assert got.tobytes() == x.tobytes()


# ----------------------------------------------------------------- skip

def _scaled_grads(rng, n, psi, scale, t):
    return [oracle.cast((rng.normal(0, 1e-3, psi) * scale).astype(np.float32), F16)
            for _ in range(n)]


@pytest.mark.parametrize("bad_value", [np.inf, -np.inf, np.nan])
def test_skip_sequence_equals_step_absent(bad_value):
    """Sixteen fp16 ranks with a loss scale of 2^16; rank 5 holds one bad
    value at iteration 3.  Iterations 1, 2 apply; 3 is skipped with nothing
    changed and the scale halved; 4.. apply with t = 3, 4, ...  The result is
    bit-identical to a run that never saw iteration 3."""
    rng = np.random.default_rng(21)
    psi, n, iters = 333, 16, 6
    S = oracle.shard_size(psi, n)
    P = n * S
    x0 = np.zeros(P, np.float32)
    x0[:psi] = rng.normal(0, 0.01, psi).astype(np.float32)

    scale, good = 2.0 ** 16, 0
    grads_by_iter = {}
    for it in range(1, iters + 1):
        grads_by_iter[it] = _scaled_grads(rng, n, psi, 2.0 ** 16, it)
    # the scale changes after the skip, so iterations after 3 are drawn at 2^15
    for it in range(4, iters + 1):
        grads_by_iter[it] = _scaled_grads(rng, n, psi, 2.0 ** 15, it)
    bad_idx = 123
    g3 = grads_by_iter[3][5].copy()
    g3[bad_idx] = oracle.cast(np.array([bad_value], np.float32), F16)[0]
    grads_by_iter[3][5] = g3

    x, m, v = x0.copy(), np.zeros(P, np.float32), np.zeros(P, np.float32)
    full = np.zeros(P, np.uint16)
    t, seen = 0, []
    for it in range(1, iters + 1):
        before = (x.tobytes(), m.tobytes(), v.tobytes(), full.tobytes())
        skipped, bad = oracle.zero_step(grads_by_iter[it], F16, psi, x, m, v, full, F16,
                                        1e-4, 0.9, 0.999, 1e-8, t + 1, loss_scale=scale)
        seen.append(skipped)
        if skipped:
            assert bad >= 1
            assert (x.tobytes(), m.tobytes(), v.tobytes(), full.tobytes()) == before
        else:
            t += 1
        scale, good = oracle.scale_update(scale, skipped, good, 2000)
        if it == 3:
            assert scale == 2.0 ** 15
    assert seen == [False, False, True, False, False, False]
    assert t == iters - 1

    # the same run without iteration 3 at all
    x2, m2, v2 = x0.copy(), np.zeros(P, np.float32), np.zeros(P, np.float32)
    full2 = np.zeros(P, np.uint16)
    t2 = 0
    for it in [1, 2, 4, 5, 6]:
        sc = 2.0 ** 16 if it < 3 else 2.0 ** 15
        skipped, _ = oracle.zero_step(grads_by_iter[it], F16, psi, x2, m2, v2, full2, F16,
                                      1e-4, 0.9, 0.999, 1e-8, t2 + 1, loss_scale=sc)
        assert not skipped
        t2 += 1
    assert x.tobytes() == x2.tobytes() and m.tobytes() == m2.tobytes()
    assert v.tobytes() == v2.tobytes() and full.tobytes() == full2.tobytes()


def test_unscaled_step_is_the_scaled_step_divided():
    """Loss scaling by a power of two is exact: grads times 2^16 with the
    scale 2^16 give the same update as the plain grads without scaling."""
    rng = np.random.default_rng(22)
    psi, n = 1000, 8
    S = oracle.shard_size(psi, n)
    P = n * S
    g32 = [rng.normal(0, 1e-3, psi).astype(np.float32) for _ in range(n)]
    plain = [oracle.cast(g, F16) for g in g32]
    scaled = [oracle.cast(g * np.float32(2 ** 16), F16) for g in g32]
    # fp16 keeps 11 bits at any normal exponent, so scaling commutes with
    # rounding except for values that were subnormal before scaling
    keep = np.ones(psi, bool)
    for g in g32:
        keep &= np.abs(g) >= 2.0 ** -14
    for lst in (plain, scaled):
        for a in lst:
            a[~keep] = 0
    xa = np.zeros(P, np.float32)
    xa[:psi] = rng.normal(0, 0.01, psi).astype(np.float32)
    xb = xa.copy()
    z = lambda: np.zeros(P, np.float32)  # noqa: E731
    ma, va, mb, vb = z(), z(), z(), z()
    fa, fb = np.zeros(P, np.uint16), np.zeros(P, np.uint16)
    oracle.zero_step(plain, F16, psi, xa, ma, va, fa, F16, 1e-3, 0.9, 0.999, 1e-8, 1)
    oracle.zero_step(scaled, F16, psi, xb, mb, vb, fb, F16, 1e-3, 0.9, 0.999, 1e-8, 1,
                     loss_scale=2.0 ** 16)
    assert xa.tobytes() == xb.tobytes() and fa.tobytes() == fb.tobytes()


def test_overflow_verdict_is_taken_on_the_unscaled_mean():
    """The verdict tests the grad the update would use (sum, /N, /scale),
    so it follows from IEEE binary32 range alone: a finite sum whose
    unscale leaves the range skips (scale 2^-8), the same sum at scale 1
    does not, finite bf16 grads whose fp32 sum leaves the range skip, and
    a non-power-of-two scale divides (the step at scale 3000 on grads
    3000 g equals the plain step on g wherever the unscaled mean comes back
    exactly)."""
    psi, n = 64, 4
    S = oracle.shard_size(psi, n)
    P = n * S

    def step(grads, gdt, scale):
        x = np.zeros(P, np.float32)
        x[:psi] = 0.5
        m, v = np.zeros(P, np.float32), np.zeros(P, np.float32)
        full = np.zeros(P, np.uint16)
        skipped, bad = oracle.zero_step(grads, gdt, psi, x, m, v, full, BF16, 1e-3, 0.9,
                                        0.999, 1e-8, 1, loss_scale=scale)
        return skipped, bad, x

    g = [np.full(psi, 1e-3, np.float32) for _ in range(n)]
    for a in g:
        a[9] = 2.0 ** 120                      # sum 2^122: finite
    assert step(g, F32, 2.0 ** -8)[:2] == (True, 1)      # 2^120 * 2^8 = 2^128: inf
    assert step(g, F32, 1.0)[:2] == (False, 0)
    assert step(g, F32, 2.0 ** -2)[:2] == (False, 0)      # 2^122: still finite
    big = [oracle.cast(np.full(psi, 1e-3, np.float32), BF16) for _ in range(n)]
    for a in big:
        a[17] = oracle.cast(np.array([2.0 ** 127], np.float32), BF16)[0]
    assert step(big, BF16, 2.0 ** 10)[:2] == (True, 1)   # 2^127 + 2^127 = inf in fp32
    base = [np.float32(1e-3) * np.arange(1, psi + 1, dtype=np.float32) for _ in range(n)]
    scaled = [a * np.float32(3000.0) for a in base]
    s1, _, x1 = step(base, F32, 0.0)
    s2, _, x2 = step(scaled, F32, 3000.0)
    assert not s1 and not s2
    # wherever the scaled mean divides back to the plain mean exactly, the
    # two steps agree element for element
    acc1, acc2 = base[0].copy(), scaled[0].copy()
    for a, b in zip(base[1:], scaled[1:]):
        acc1 = acc1 + a
        acc2 = acc2 + b
    sums_ok = ((acc2 / np.float32(n)) / np.float32(3000.0)) == (acc1 / np.float32(n))
    assert sums_ok.sum() > psi // 2
    assert (x1[:psi][sums_ok] == x2[:psi][sums_ok]).all()


def test_without_loss_scaling_nan_propagates():
    """Loss scaling off: no skip; a non-finite grad is reported and reaches
    the state of its element only."""
    psi, n = 64, 4
    S = oracle.shard_size(psi, n)
    grads = [np.full(psi, 0.01, np.float32) for _ in range(n)]
    grads[2][7] = np.nan
    x, m, v = np.zeros(n * S, np.float32), np.zeros(n * S, np.float32), np.zeros(n * S, np.float32)
    full = np.zeros(n * S, np.float32)
    skipped, bad = oracle.zero_step(grads, F32, psi, x, m, v, full, F32, 1e-3, 0.9, 0.999,
                                    1e-8, 1)
    assert not skipped and bad == 1
    assert np.isnan(x[7]) and np.isnan(m[7]) and np.isnan(full[7])
    assert np.isfinite(np.delete(x, 7)).all()


def test_scale_update_policy():
    s, g = oracle.scale_update(65536.0, True, 17, 2000)
    assert (s, g) == (32768.0, 0)
    s, g = oracle.scale_update(32768.0, False, 1998, 2000)
    assert (s, g) == (32768.0, 1999)
    s, g = oracle.scale_update(32768.0, False, 1999, 2000)
    assert (s, g) == (65536.0, 0)


def test_scale_update_equals_torch_grad_scaler():
    """The loss-scale policy against a library routine: PyTorch's GradScaler
    update (backoff 0.5 on a non-finite step, growth x2 after growth_interval
    clean steps, never growing to infinity), over random sequences of
    skipped and clean steps, from ordinary and extreme scales."""
    import torch
    rng = np.random.default_rng(5)
    fmax = float(np.finfo(np.float32).max)
    starts = [65536.0, 1.0, 2.0 ** -140, 2.0 ** 126, fmax / 2, 3.0]
    for trial in range(60):
        interval = int(rng.integers(1, 6))
        s0 = starts[trial % len(starts)]
        s_o, g_o = s0, 0
        s_t = torch.tensor([s0], dtype=torch.float32)
        g_t = torch.tensor([0], dtype=torch.int32)
        for _ in range(40):
            skipped = bool(rng.random() < 0.3)
            s_o, g_o = oracle.scale_update(s_o, skipped, g_o, interval)
            torch._amp_update_scale_(s_t, g_t, torch.tensor([1.0 if skipped else 0.0]),
                                     2.0, 0.5, interval)
            assert np.float32(s_o).tobytes() == s_t.numpy().tobytes(), (trial, s_o, s_t)
            assert g_o == int(g_t.item())
