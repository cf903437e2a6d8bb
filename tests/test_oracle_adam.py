"""Pins of the oracle's Adam and of the composed ZeRO step.

Adam as in "ZeRO 与 FSDP：切分优化器状态、梯度与参数", section 从零实现 ZeRO
的 Adam (ZeroAdam.step: m, v with bias correction, eps outside the root);
the 4-process check and its printed outcome are from the same section.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import BF16, F16, F32

U = 2.0 ** -24  # unit roundoff of binary32


def _fresh(n, rng, sigma=0.01):
    x = rng.normal(0, sigma, n).astype(np.float32)
    return x, np.zeros(n, np.float32), np.zeros(n, np.float32)


@pytest.mark.parametrize("lr,b1,b2,eps", [(1e-2, 0.9, 0.999, 1e-8), (3e-4, 0.8, 0.95, 1e-6)])
def test_first_step_closed_form(lr, b1, b2, eps):
    """m = v = 0, t = 1: m_hat = g and v_hat = g^2, so the step is
    lr * g / (|g| + eps), about lr * sign(g) for |g| >> eps."""
    rng = np.random.default_rng(10)
    x, m, v = _fresh(4096, rng)
    g = rng.normal(0, 1e-3, 4096).astype(np.float32)
    x0 = x.copy()
    oracle.adam(x, m, v, g, lr, b1, b2, eps, 1)
    gd = g.astype(np.float64)
    want = x0.astype(np.float64) - lr * gd / (np.abs(gd) + eps)
    upd = np.abs(lr * gd / (np.abs(gd) + eps))
    # about ten roundings on the update, one on the subtraction
    bound = 12 * U * upd + np.spacing(np.abs(want).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(x.astype(np.float64) - want) <= bound)
    # |g| >> eps: the step is lr * sign(g) to within eps/|g|
    big = np.abs(gd) > 1e3 * eps
    step = (x0.astype(np.float64) - x.astype(np.float64))[big]
    assert np.allclose(step, lr * np.sign(gd[big]), rtol=2e-3, atol=0)
    assert np.array_equal(np.sign(x0 - x)[g != 0], np.sign(g)[g != 0])


def test_eps_outside_the_root():
    """With |g| = eps the first step is exactly half of lr (eps added after
    the square root); eps inside the root would give lr / sqrt(1 + 1/eps)."""
    eps = float(np.float32(1e-3))   # exactly representable in both widths
    g = np.full(8, eps, np.float32)
    x = np.zeros(8, np.float32)
    m = np.zeros(8, np.float32)
    v = np.zeros(8, np.float32)
    oracle.adam(x, m, v, g, 1.0, 0.5, 0.5, eps, 1)
    assert np.allclose(x, -0.5, rtol=8 * U, atol=0)


def test_zero_gradient_is_a_fixed_point():
    rng = np.random.default_rng(11)
    x, m, v = _fresh(1000, rng)
    x0 = x.copy()
    for t in range(1, 6):
        oracle.adam(x, m, v, np.zeros(1000, np.float32), 1e-2, 0.9, 0.999, 1e-8, t)
    assert x.tobytes() == x0.tobytes()
    assert not m.any() and not v.any()


@pytest.mark.parametrize("b1,b2", [(0.9, 0.999), (0.5, 0.75), (0.99, 0.9999)])
def test_constant_gradient_every_step_is_the_same(b1, b2):
    """With the same g every step, m_t = g (1 - b1^t) and v_t = g^2 (1 - b2^t)
    exactly, so bias correction gives m_hat = g, v_hat = g^2 at every t and
    each step moves x by lr * g / (|g| + eps).  A wrong exponent in a bias
    correction, or a missing (1 - beta) weight, breaks this."""
    rng = np.random.default_rng(12)
    n, T, lr, eps = 2048, 25, 1e-3, 1e-8
    x, m, v = _fresh(n, rng)
    g = rng.normal(0, 1e-2, n).astype(np.float32)
    x0 = x.astype(np.float64)
    for t in range(1, T + 1):
        oracle.adam(x, m, v, g, lr, b1, b2, eps, t)
        s = oracle.adam_scalars(b1, b2, t)
        mh = m.astype(np.float64) / np.float64(s[2])
        assert np.allclose(mh, g, rtol=16 * t * U, atol=0)
    gd = g.astype(np.float64)
    want = x0 - T * lr * gd / (np.abs(gd) + eps)
    err = np.abs(x.astype(np.float64) - want)
    assert np.all(err <= T * (12 * U * lr + 2 * U * np.abs(want)))


def _round_f32(q: Fraction) -> np.float32:
    """Nearest binary32 to an exact rational (ties to even)."""
    f = np.float32(float(q))
    cands = [f, np.nextafter(f, np.float32(np.inf)), np.nextafter(f, np.float32(-np.inf))]
    best = min(cands, key=lambda c: (abs(Fraction(float(c)) - q),
                                      int(np.float32(c).view(np.uint32)) & 1))
    return np.float32(best)


def test_adam_scalars_against_exact_rationals():
    for b1, b2 in [(0.9, 0.999), (0.95, 0.98)]:
        f1, f2 = Fraction(b1), Fraction(b2)   # the doubles the caller passes
        for t in list(range(1, 40)) + [100, 1000, 4096]:
            s = oracle.adam_scalars(b1, b2, t)
            assert s[0] == _round_f32(1 - f1)
            assert s[1] == _round_f32(1 - f2)
            assert s[2] == _round_f32(1 - f1 ** t), t
            assert s[3] == _round_f32(1 - f2 ** t), t


def test_against_torch_adam():
    """torch.optim.Adam (a library routine) on the same gradient sequence:
    different rounding order, same method, so agreement to a few ulps."""
    rng = np.random.default_rng(13)
    n, T, lr = 5000, 10, 1e-2
    x, m, v = _fresh(n, rng)
    p = torch.nn.Parameter(torch.from_numpy(x.copy()))
    opt = torch.optim.Adam([p], lr=lr, betas=(0.9, 0.999), eps=1e-8, foreach=False)
    gmax = 0.0
    for t in range(1, T + 1):
        g = rng.normal(0, 1e-2, n).astype(np.float32)
        gmax = max(gmax, float(np.abs(g).max()))
        oracle.adam(x, m, v, g, lr, 0.9, 0.999, 1e-8, t)
        p.grad = torch.from_numpy(g.copy())
        opt.step()
    st = opt.state[p]
    diff = np.abs(x - p.detach().numpy())
    assert diff.max() < 1e-5                      # the pages' bar
    assert diff.max() <= 64 * U * T * lr          # a few ulps of the step size
    # m sums terms of both signs: compare against the scale of the terms
    np.testing.assert_allclose(m, st["exp_avg"].numpy(), rtol=0, atol=16 * T * U * gmax)
    np.testing.assert_allclose(v, st["exp_avg_sq"].numpy(), rtol=4 * T * U, atol=0)


def test_sharded_equals_unsharded_bit_exact():
    """ZeRO-2 sharded step == plain Adam over the whole vector on the
    all-reduced mean grad, bit for bit (the update is elementwise), for the
    all-ranks composition and for each rank's own view."""
    rng = np.random.default_rng(14)
    for psi, n, gd, pd in [(19210, 4, F32, F32), (1001, 8, BF16, BF16), (77, 16, F16, F16),
                           (5, 8, BF16, F32)]:
        S = oracle.shard_size(psi, n)
        P = n * S
        x0 = np.zeros(P, np.float32)
        x0[:psi] = rng.normal(0, 0.01, psi).astype(np.float32)
        xa, ma, va = x0.copy(), np.zeros(P, np.float32), np.zeros(P, np.float32)
        xb, mb, vb = x0.copy(), np.zeros(P, np.float32), np.zeros(P, np.float32)
        xc, mc, vc = x0.copy(), np.zeros(P, np.float32), np.zeros(P, np.float32)
        full = np.zeros(P, oracle.NP_STORAGE[pd])
        full_c = np.zeros(P, oracle.NP_STORAGE[pd])
        for t in range(1, 4):
            g32 = [rng.normal(0, 1e-3, psi).astype(np.float32) for _ in range(n)]
            grads = g32 if gd == F32 else [oracle.cast(g, gd) for g in g32]
            skipped, bad = oracle.zero_step(grads, gd, psi, xa, ma, va, full, pd,
                                            1e-2, 0.9, 0.999, 1e-8, t)
            assert not skipped and bad == 0
            gmean = oracle.all_reduce_mean(grads, gd, psi)
            oracle.adam(xb, mb, vb, gmean, 1e-2, 0.9, 0.999, 1e-8, t)
            for r in range(n):
                sl = slice(r * S, (r + 1) * S)
                padded = [np.concatenate([g, np.zeros(P - psi, g.dtype)]) for g in grads]
                slices = [np.ascontiguousarray(g[sl]) for g in padded]
                lp = np.zeros(S, oracle.NP_STORAGE[pd])
                xr, mr, vr = xc[sl].copy(), mc[sl].copy(), vc[sl].copy()
                oracle.zero_rank_step(slices, gd, psi, r, xr, mr, vr, lp, pd,
                                      1e-2, 0.9, 0.999, 1e-8, t)
                xc[sl], mc[sl], vc[sl] = xr, mr, vr
                full_c[sl] = lp
        for a, b in [(xa, xb), (ma, mb), (va, vb), (xa, xc), (ma, mc), (va, vc)]:
            assert a.tobytes() == b.tobytes()
        assert full.tobytes() == oracle.cast(xb, pd).tobytes() == full_c.tobytes()
        # the padding stays exactly +0 everywhere
        for a in (xa, ma, va):
            assert not a[psi:].any() and not np.signbit(a[psi:]).any()


def test_pages_four_rank_mlp_check():
    """The pages' zero_check: an MLP Linear(64,256)+GELU+Linear(256,10), 4
    ranks each on a quarter of a batch of 32, 3 Adam steps with lr 1e-2,
    against single-process torch.optim.Adam on the full batch: every
    parameter agrees to better than 1e-5 (printed: True)."""
    golden = {}
    with open(os.path.join(os.path.dirname(__file__), "golden", "zero_adam_check.txt"),
              encoding="utf-8") as f:
        for ln in f:
            if ln.strip() and not ln.startswith("#"):
                k, val = ln.split()
                golden[k] = val
    world, steps, lr = int(golden["world"]), int(golden["steps"]), float(golden["lr"])
    batch = int(golden["batch"])

    def make():
        torch.manual_seed(0)
        return torch.nn.Sequential(torch.nn.Linear(64, 256), torch.nn.GELU(),
                                   torch.nn.Linear(256, 10))

    torch.manual_seed(123)
    X, Y = torch.randn(batch, 64), torch.randint(0, 10, (batch,))
    loss_fn = torch.nn.CrossEntropyLoss()
    ref, model = make(), make()
    opt_ref = torch.optim.Adam(ref.parameters(), lr=lr)
    params = list(model.parameters())
    numel = sum(p.numel() for p in params)
    assert numel == int(golden["numel"])
    S = oracle.shard_size(numel, world)
    P = world * S
    master = np.zeros(P, np.float32)
    master[:numel] = torch.cat([p.detach().flatten() for p in params]).numpy()
    m, v = np.zeros(P, np.float32), np.zeros(P, np.float32)
    full = np.zeros(P, np.float32)
    for t in range(1, steps + 1):
        opt_ref.zero_grad()
        loss_fn(ref(X), Y).backward()
        opt_ref.step()
        grads = []
        for r in range(world):
            model.zero_grad()
            loc = slice(r * batch // world, (r + 1) * batch // world)
            loss_fn(model(X[loc]), Y[loc]).backward()
            grads.append(torch.cat([p.grad.flatten() for p in params]).numpy().copy())
        skipped, _ = oracle.zero_step(grads, F32, numel, master, m, v, full, F32,
                                      lr, 0.9, 0.999, 1e-8, t)
        assert not skipped
        off = 0
        with torch.no_grad():
            for p in params:
                p.copy_(torch.from_numpy(full[off:off + p.numel()]).view_as(p))
                off += p.numel()
    diff = max((a - b).abs().max().item() for a, b in zip(ref.parameters(), model.parameters()))
    assert diff < float(golden["max_abs_diff_below"])
    assert oracle.memory.zero_adam_state_bytes(numel, world) == int(golden["state_bytes_rank"])


# ------------------------------------------------------------------ AdamW

def test_adamw_zero_gradient_is_pure_decay():
    """AdamW with g = 0: m = v = 0, the Adam step is exactly 0, and each step
    multiplies x by d = fp32(1 - lr*wd): x_t is t exact fp32 products."""
    rng = np.random.default_rng(30)
    x, m, v = _fresh(1000, rng)
    x0 = x.copy()
    lr, wd = 1e-2, 0.1
    d = np.float32(1.0 - lr * wd)
    want = x0.copy()
    for t in range(1, 8):
        oracle.adam(x, m, v, np.zeros(1000, np.float32), lr, 0.9, 0.999, 1e-8, t,
                    weight_decay=wd)
        want = (want * d).astype(np.float32)
    assert x.tobytes() == want.tobytes()
    assert np.allclose(x, x0.astype(np.float64) * (1 - lr * wd) ** 7, rtol=8 * U, atol=0)


def test_adamw_without_decay_is_adam_bit_for_bit():
    rng = np.random.default_rng(31)
    xa, ma, va = _fresh(3000, rng)
    xb, mb, vb = xa.copy(), ma.copy(), va.copy()
    for t in range(1, 5):
        g = rng.normal(0, 1e-2, 3000).astype(np.float32)
        oracle.adam(xa, ma, va, g, 1e-3, 0.9, 0.999, 1e-8, t)
        oracle.adam(xb, mb, vb, g, 1e-3, 0.9, 0.999, 1e-8, t, weight_decay=0.0)
    assert xa.tobytes() == xb.tobytes()


def test_adamw_against_torch():
    """torch.optim.AdamW (library): decay first, then the Adam step."""
    rng = np.random.default_rng(32)
    n, T, lr, wd = 5000, 10, 1e-2, 0.05
    x, m, v = _fresh(n, rng, sigma=0.5)
    p = torch.nn.Parameter(torch.from_numpy(x.copy()))
    opt = torch.optim.AdamW([p], lr=lr, betas=(0.9, 0.999), eps=1e-8, weight_decay=wd,
                            foreach=False)
    for t in range(1, T + 1):
        g = rng.normal(0, 1e-2, n).astype(np.float32)
        oracle.adam(x, m, v, g, lr, 0.9, 0.999, 1e-8, t, weight_decay=wd)
        p.grad = torch.from_numpy(g.copy())
        opt.step()
    got, want = x.astype(np.float64), p.detach().numpy().astype(np.float64)
    assert np.abs(got - want).max() <= 64 * U * T * (lr + np.abs(want).max() * lr * wd)
    # and the decay is really applied: far from plain Adam's result
    y, my, vy = _fresh(n, np.random.default_rng(32), sigma=0.5)
    rng2 = np.random.default_rng(32)
    _fresh(n, rng2, sigma=0.5)
    for t in range(1, T + 1):
        oracle.adam(y, my, vy, rng2.normal(0, 1e-2, n).astype(np.float32), lr, 0.9, 0.999,
                    1e-8, t)
    assert np.abs(y - x).max() > 100 * np.abs(got - want).max()
