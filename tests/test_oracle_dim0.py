"""Pins of the oracle's per-parameter dim-0 layout (FSDP2), from "ZeRO 与
FSDP：切分优化器状态、梯度与参数", section ZeRO-3 与 FSDP."""
import os

import numpy as np
import torch

import oracle
from oracle import F32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fsdp2_check.txt")


def test_chunks_match_torch_chunk():
    """Rank r holds rows [r*c, r*c + c) with c = ceil(rows/N); the valid rows
    per rank are torch.chunk's chunks, empty ones included for ranks past
    the end."""
    for rows in range(0, 41):
        for n in range(1, 10):
            S = oracle.row_shard_size(rows, 3, n)
            c = S // 3
            chunks = torch.chunk(torch.arange(rows), n) if rows else ()
            for r in range(n):
                want = len(chunks[r]) if r < len(chunks) else 0
                assert max(0, min(c, rows - r * c)) == want, (rows, n, r)
            assert c * n >= rows and (c - 1) * n < max(rows, 1)


def test_pages_fsdp2_check():
    g = dict(ln.split(None, 1) for ln in open(GOLDEN, encoding="utf-8")
             if ln.strip() and not ln.startswith("#"))
    world, steps, lr, batch = int(g["world"]), int(g["steps"]), float(g["lr"]), int(g["batch"])

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
    # one unit per parameter, sharded along dim 0
    units = []
    for p in params:
        rows = p.shape[0]
        row = p.numel() // rows
        S = oracle.row_shard_size(rows, row, world)
        units.append((rows, row, S))
    rows, row, S = units[0]
    assert tuple(int(x) for x in g["first_weight_full"].split()) == (rows, row)
    assert (S // row, row) == tuple(int(x) for x in g["first_weight_local"].split())
    state = {}
    for u, (p, (rows, row, S)) in enumerate(zip(params, units)):
        flat = np.zeros(S * world, np.float32)
        flat[:p.numel()] = p.detach().flatten().numpy()
        for r in range(world):
            state[u, r] = [flat[r * S:(r + 1) * S].copy(), np.zeros(S, np.float32),
                           np.zeros(S, np.float32)]
    for t in range(1, steps + 1):
        opt_ref.zero_grad()
        loss_fn(ref(X), Y).backward()
        opt_ref.step()
        local = []
        for r in range(world):
            model.zero_grad()
            sl = slice(r * batch // world, (r + 1) * batch // world)
            loss_fn(model(X[sl]), Y[sl]).backward()
            local.append([p.grad.flatten().numpy().copy() for p in params])
        with torch.no_grad():
            for u, (p, (rows, row, S)) in enumerate(zip(params, units)):
                padded = []
                for r in range(world):
                    f = np.zeros(S * world, np.float32)
                    f[:p.numel()] = local[r][u]
                    padded.append(f)
                shards = []
                for r in range(world):
                    slices = [np.ascontiguousarray(f[r * S:(r + 1) * S]) for f in padded]
                    x, m, v = state[u, r]
                    lp = np.zeros(S, np.float32)
                    skipped, _ = oracle.zero_rank_step(slices, F32, p.numel(), r, x, m, v, lp,
                                                       F32, lr, 0.9, 0.999, 1e-8, t, shard=S)
                    assert not skipped
                    shards.append(lp)
                full = oracle.all_gather(shards, F32)
                p.copy_(torch.from_numpy(full[:p.numel()]).view_as(p))
    diff = max((a - b).abs().max().item() for a, b in zip(ref.parameters(), model.parameters()))
    assert diff < float(g["max_abs_diff_below"])


def test_dim0_step_equals_unsharded_adam():
    """Any shard length (here whole rows) leaves the elementwise step equal
    to plain Adam on the mean grad, bit for bit, padding rows at +0."""
    rng = np.random.default_rng(40)
    rows, row, world = 10, 7, 4
    numel = rows * row
    S = oracle.row_shard_size(rows, row, world)       # 3 rows = 21 elements
    assert S == 21 and S * world == 84
    x0 = np.zeros(S * world, np.float32)
    x0[:numel] = rng.normal(0, 0.01, numel)
    xa, ma, va = x0.copy(), np.zeros_like(x0), np.zeros_like(x0)
    xb, mb, vb = x0.copy(), np.zeros_like(x0), np.zeros_like(x0)
    full = np.zeros(S * world, np.float32)
    for t in (1, 2, 3):
        grads = [rng.normal(0, 1e-3, numel).astype(np.float32) for _ in range(world)]
        oracle.zero_step(grads, F32, numel, xa, ma, va, full, F32, 1e-3, 0.9, 0.999, 1e-8, t,
                         shard=S)
        acc = oracle.rank_sum([np.concatenate([g, np.zeros(S * world - numel, np.float32)])
                               for g in grads], F32, S * world, numel)
        gm, _ = oracle.average(acc, world)
        oracle.adam(xb, mb, vb, gm, 1e-3, 0.9, 0.999, 1e-8, t)
    assert xa.tobytes() == xb.tobytes() and full.tobytes() == xa.tobytes()
    assert not xa[numel:].any()
