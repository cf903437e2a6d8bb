"""ShardedZeroAdam, the pages' ZeroAdam with one process per rank, on the
pages' own check ("ZeRO 与 FSDP…", 从零实现 ZeRO 的 Adam: four gloo processes
train the MLP Linear(64,256)+GELU+Linear(256,10) with equal local batches).
Four processes share this GPU (their data moves through host memory; no
kernel of one waits for another).  Every rank's model must end within the
pages' 1e-5 of torch.optim.Adam on the full batch, every rank must report
the pages' 57,636 bytes of state, and the final parameters must equal, bit
for bit, what the oracle's all-ranks step computes from the four ranks'
saved gradients."""
import os

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from tests.test_multiprocess_gloo import _free_port

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
WORLD, PER_RANK, LR, STEPS = 4, 8, 1e-2, 5


def _flat(params):
    return torch.cat([p.detach().reshape(-1).float().cpu() for p in params]).numpy()


def _rank(rank, port, out_dir, bucket_elems=0):
    import copy
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import zero_sharded_optimizer_step_gb300 as z
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    torch.cuda.set_device(0)
    dev = torch.device("cuda:0")
    torch.manual_seed(0)                       # the same model on every rank
    model = torch.nn.Sequential(torch.nn.Linear(64, 256), torch.nn.GELU(),
                                torch.nn.Linear(256, 10)).to(dev)
    ref = copy.deepcopy(model)
    init = _flat(model.parameters())
    opt = z.ShardedZeroAdam(model.parameters(), lr=LR, betas=(0.9, 0.999), eps=1e-8,
                            bucket_elems=bucket_elems)
    ref_opt = torch.optim.Adam(ref.parameters(), lr=LR, betas=(0.9, 0.999), eps=1e-8)
    loss_fn = torch.nn.CrossEntropyLoss()
    grads = []
    for it in range(STEPS):
        gen = torch.Generator().manual_seed(100 + it)   # the same batch on every rank
        x = torch.randn(WORLD * PER_RANK, 64, generator=gen).to(dev)
        y = torch.randint(0, 10, (WORLD * PER_RANK,), generator=gen).to(dev)
        sl = slice(rank * PER_RANK, (rank + 1) * PER_RANK)
        opt.zero_grad()
        if bucket_elems:
            # this rank's grads, for the oracle, from an identical backward of
            # a copy (the bucketed optimizer consumes and frees .grad)
            twin = copy.deepcopy(model)
            loss_fn(twin(x[sl]), y[sl]).backward()
            grads.append(torch.cat([p.grad.reshape(-1) for p in twin.parameters()]).cpu().numpy())
            loss_fn(model(x[sl]), y[sl]).backward()
            # the buckets were exchanged during the backward; no grad is kept
            assert all(p.grad is None for p in model.parameters())
        else:
            loss_fn(model(x[sl]), y[sl]).backward()
            grads.append(torch.cat([p.grad.reshape(-1)
                                    for p in model.parameters()]).cpu().numpy())
        assert opt.step() is False
        ref_opt.zero_grad(set_to_none=True)
        loss_fn(ref(x), y).backward()
        ref_opt.step()
    torch.cuda.synchronize()
    worst = max((a - b).abs().max().item() for a, b in zip(model.parameters(), ref.parameters()))
    np.savez(os.path.join(out_dir, "rank%d.npz" % rank), init=init,
             final=_flat(model.parameters()), grads=np.stack(grads), worst=worst,
             numel=opt.numel, state_bytes=opt.state_bytes())
    opt.close()
    dist.destroy_process_group()


@pytest.mark.parametrize("bucket_elems", [0, 4_000])
def test_sharded_zero_adam_trains_the_pages_mlp(bucket_elems):
    """bucket_elems > 0: the grads exchanged bucket by bucket during the
    backward (5 buckets of the 19,212-element vector, across parameter and
    shard boundaries) -- the same result bit for bit."""
    import tempfile

    import oracle
    with tempfile.TemporaryDirectory() as out:
        mp.start_processes(_rank, args=(_free_port(), out, bucket_elems), nprocs=WORLD,
                           join=True, start_method="spawn")
        ranks = [np.load(os.path.join(out, "rank%d.npz" % r)) for r in range(WORLD)]
    for d in ranks:
        assert int(d["numel"]) == 19_210
        assert int(d["state_bytes"]) == 57_636       # the pages' printed per-rank figure
        assert float(d["worst"]) < 1e-5, float(d["worst"])
        assert d["init"].tobytes() == ranks[0]["init"].tobytes()
    # the oracle's all-ranks step on the ranks' own gradients
    numel = 19_210
    P = oracle.shard_size(numel, WORLD) * WORLD
    x = np.zeros(P, np.float32)
    x[:numel] = ranks[0]["init"]
    m, v = np.zeros(P, np.float32), np.zeros(P, np.float32)
    full = np.zeros(P, np.float32)
    for it in range(STEPS):
        g = [np.ascontiguousarray(d["grads"][it], np.float32) for d in ranks]
        oracle.zero_step(g, oracle.F32, numel, x, m, v, full, oracle.F32, LR, 0.9, 0.999, 1e-8,
                         it + 1)
    for r, d in enumerate(ranks):
        assert d["final"].tobytes() == full[:numel].tobytes(), r


def _rank_fp16(rank, port, out_dir, bucket_elems):
    """The MLP in fp16 with loss scaling: the loss is multiplied by the
    optimizer's current scale; rank 1 plants a +inf in one grad element at
    step 2 (a tensor hook, before accumulation), which must skip the step on
    every rank and halve the scale."""
    import copy
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import zero_sharded_optimizer_step_gb300 as z
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    world = 2
    dist.init_process_group("gloo", rank=rank, world_size=world)
    torch.cuda.set_device(0)
    dev = torch.device("cuda:0")
    torch.manual_seed(0)
    model = torch.nn.Sequential(torch.nn.Linear(64, 256), torch.nn.GELU(),
                                torch.nn.Linear(256, 10)).to(dev).half()
    init = _flat(model.parameters())
    opt = z.ShardedZeroAdam(model.parameters(), lr=LR, betas=(0.9, 0.999), eps=1e-8,
                            loss_scale=1024.0, bucket_elems=bucket_elems)
    first = next(iter(model.parameters()))
    plant = {"on": False}

    def inf_hook(g):
        if plant["on"]:
            g = g.clone()
            g.view(-1)[5] = float("inf")
        return g
    first.register_hook(inf_hook)
    loss_fn = torch.nn.CrossEntropyLoss()
    grads, skips, scales = [], [], []
    for it in range(4):
        gen = torch.Generator().manual_seed(200 + it)
        x = torch.randn(world * PER_RANK, 64, generator=gen).to(dev).half()
        y = torch.randint(0, 10, (world * PER_RANK,), generator=gen).to(dev)
        sl = slice(rank * PER_RANK, (rank + 1) * PER_RANK)
        plant["on"] = rank == 1 and it == 1
        scales.append(opt.scale)
        opt.zero_grad()
        twin = copy.deepcopy(model)              # the same backward, for the record
        twin_first = next(iter(twin.parameters()))
        twin_first.register_hook(inf_hook)
        (loss_fn(twin(x[sl]).float(), y[sl]) * opt.scale).backward()
        grads.append(torch.cat([p.grad.reshape(-1) for p in twin.parameters()])
                     .cpu().view(torch.int16).numpy().view(np.uint16))
        (loss_fn(model(x[sl]).float(), y[sl]) * opt.scale).backward()
        skips.append(opt.step())
    torch.cuda.synchronize()
    final = torch.cat([p.detach().reshape(-1) for p in model.parameters()]).cpu()
    np.savez(os.path.join(out_dir, "rank%d.npz" % rank), init=init, grads=np.stack(grads),
             skips=np.array(skips), scales=np.array(scales),
             final=final.view(torch.int16).numpy().view(np.uint16), scale=opt.scale, t=opt.t)
    opt.close()
    dist.destroy_process_group()


@pytest.mark.parametrize("bucket_elems", [0, 5_000])
def test_sharded_zero_adam_fp16_loss_scaled_skip(bucket_elems):
    import tempfile

    import oracle
    with tempfile.TemporaryDirectory() as out:
        mp.start_processes(_rank_fp16, args=(_free_port(), out, bucket_elems), nprocs=2,
                           join=True, start_method="spawn")
        ranks = [np.load(os.path.join(out, "rank%d.npz" % r)) for r in range(2)]
    numel, world = 19_210, 2
    P = oracle.shard_size(numel, world) * world
    x = np.zeros(P, np.float32)
    x[:numel] = ranks[0]["init"]
    m, v = np.zeros(P, np.float32), np.zeros(P, np.float32)
    full = np.zeros(P, np.uint16)
    scale, good, t, skips = 1024.0, 0, 0, []
    for it in range(4):
        assert float(ranks[0]["scales"][it]) == scale
        g = [np.ascontiguousarray(d["grads"][it]) for d in ranks]
        sk, _ = oracle.zero_step(g, oracle.F16, numel, x, m, v, full, oracle.F16, LR, 0.9,
                                 0.999, 1e-8, t + 1, loss_scale=scale)
        skips.append(sk)
        if not sk:
            t += 1
        scale, good = oracle.scale_update(scale, sk, good, 2000)
    assert skips == [False, True, False, False]
    for r, d in enumerate(ranks):
        assert list(d["skips"]) == skips, r
        assert float(d["scale"]) == scale == 512.0 and int(d["t"]) == t == 3
        assert d["final"].tobytes() == full[:numel].tobytes(), r


def _rank_resume(rank, port, out_dir, bucket_elems):
    """Two steps, a checkpoint of every rank's shard, two more steps (A);
    then a fresh model and optimizer loaded from the checkpoint run the same
    two steps (B).  A and B must agree bit for bit."""
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import zero_sharded_optimizer_step_gb300 as z
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    world = 2
    dist.init_process_group("gloo", rank=rank, world_size=world)
    torch.cuda.set_device(0)
    dev = torch.device("cuda:0")
    loss_fn = torch.nn.CrossEntropyLoss()

    def build(seed):
        torch.manual_seed(seed)
        m = torch.nn.Sequential(torch.nn.Linear(64, 256), torch.nn.GELU(),
                                torch.nn.Linear(256, 10)).to(dev).half()
        o = z.ShardedZeroAdam(m.parameters(), lr=LR, betas=(0.9, 0.999), eps=1e-8,
                              loss_scale=2048.0, bucket_elems=bucket_elems)
        return m, o

    def train(model, opt, its):
        for it in its:
            gen = torch.Generator().manual_seed(300 + it)
            x = torch.randn(world * PER_RANK, 64, generator=gen).to(dev).half()
            y = torch.randint(0, 10, (world * PER_RANK,), generator=gen).to(dev)
            sl = slice(rank * PER_RANK, (rank + 1) * PER_RANK)
            opt.zero_grad()
            (loss_fn(model(x[sl]).float(), y[sl]) * opt.scale).backward()
            opt.step()

    model, opt = build(0)
    train(model, opt, [0, 1])
    sd = opt.state_dict()
    sd = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in sd.items()}   # as if saved
    train(model, opt, [2, 3])
    a = torch.cat([p.detach().reshape(-1) for p in model.parameters()]).cpu()
    ax = opt.state()[0].cpu()
    model2, opt2 = build(1)                     # other initial weights: all must come back
    opt2.load_state_dict(sd)
    train(model2, opt2, [2, 3])
    b = torch.cat([p.detach().reshape(-1) for p in model2.parameters()]).cpu()
    bx = opt2.state()[0].cpu()
    np.savez(os.path.join(out_dir, "rank%d.npz" % rank),
             a=a.view(torch.int16).numpy(), b=b.view(torch.int16).numpy(),
             ax=ax.numpy(), bx=bx.numpy(), ta=opt.t, tb=opt2.t, sa=opt.scale, sb=opt2.scale)
    opt.close()
    opt2.close()
    dist.destroy_process_group()


@pytest.mark.parametrize("bucket_elems", [0, 6_000])
def test_sharded_zero_adam_resumes_from_its_state(bucket_elems):
    import tempfile
    with tempfile.TemporaryDirectory() as out:
        mp.start_processes(_rank_resume, args=(_free_port(), out, bucket_elems), nprocs=2,
                           join=True, start_method="spawn")
        ranks = [np.load(os.path.join(out, "rank%d.npz" % r)) for r in range(2)]
    for d in ranks:
        assert d["a"].tobytes() == d["b"].tobytes()
        assert d["ax"].tobytes() == d["bx"].tobytes()
        assert int(d["ta"]) == int(d["tb"]) == 4 and float(d["sa"]) == float(d["sb"])
    assert ranks[0]["a"].tobytes() == ranks[1]["a"].tobytes()


def _mlp(dev, seed):
    torch.manual_seed(seed)
    return torch.nn.Sequential(torch.nn.Linear(64, 256), torch.nn.GELU(),
                               torch.nn.Linear(256, 10)).to(dev)


def _train_steps(model, opt, rank, world, its, dev):
    """The pages' data-parallel step: every rank the same global batch,
    its own slice of it; returns this rank's local grads of each step."""
    loss_fn = torch.nn.CrossEntropyLoss()
    grads = []
    for it in its:
        gen = torch.Generator().manual_seed(500 + it)
        x = torch.randn(4 * PER_RANK, 64, generator=gen).to(dev)
        y = torch.randint(0, 10, (4 * PER_RANK,), generator=gen).to(dev)
        per = 4 * PER_RANK // world
        sl = slice(rank * per, (rank + 1) * per)
        opt.zero_grad()
        loss_fn(model(x[sl]), y[sl]).backward()
        grads.append(torch.cat([p.grad.reshape(-1) for p in model.parameters()]).cpu().numpy())
        assert opt.step() is False
    return grads


def _rank_reshard(rank, world, port, out_dir, phase):
    """Phase "save": two ranks train two steps and save their shards.  Phase
    "resume": four ranks start from other weights, load the two-rank
    checkpoint resharded for four, and train two more steps."""
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import zero_sharded_optimizer_step_gb300 as z
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    torch.cuda.set_device(0)
    dev = torch.device("cuda:0")
    if phase == "save":
        model = _mlp(dev, 0)
        opt = z.ShardedZeroAdam(model.parameters(), lr=LR, betas=(0.9, 0.999), eps=1e-8)
        _train_steps(model, opt, rank, world, [0, 1], dev)
        sd = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in opt.state_dict().items()}
        torch.save(sd, os.path.join(out_dir, "ckpt%d.pt" % rank))
        np.save(os.path.join(out_dir, "saved_params%d.npy" % rank), _flat(model.parameters()))
    else:
        model = _mlp(dev, 1)                    # other weights: all must come from the checkpoint
        opt = z.ShardedZeroAdam(model.parameters(), lr=LR, betas=(0.9, 0.999), eps=1e-8)
        full = z.consolidate_state([torch.load(os.path.join(out_dir, "ckpt%d.pt" % r))
                                    for r in range(2)])
        opt.load_state_dict(z.shard_state(full, world, rank))
        loaded = _flat(model.parameters())
        grads = _train_steps(model, opt, rank, world, [2, 3], dev)
        np.savez(os.path.join(out_dir, "resume%d.npz" % rank), loaded=loaded,
                 grads=np.stack(grads), final=_flat(model.parameters()),
                 master=opt.state()[0].cpu().numpy(), t=opt.t)
    opt.close()
    dist.destroy_process_group()


def test_checkpoint_resumes_on_another_rank_count(tmp_path):
    """A two-rank checkpoint, consolidated and resharded, resumes on four
    ranks: every rank's parameters come back as saved, and the next two
    steps equal, bit for bit, the oracle's all-ranks steps from the
    consolidated state on the four ranks' gradients."""
    import oracle

    import zero_sharded_optimizer_step_gb300 as z
    for world, phase in ((2, "save"), (4, "resume")):
        mp.start_processes(_rank_reshard, args=(world, _free_port(), str(tmp_path), phase),
                           nprocs=world, join=True, start_method="spawn")
    saved = np.load(os.path.join(tmp_path, "saved_params0.npy"))
    assert saved.tobytes() == np.load(os.path.join(tmp_path, "saved_params1.npy")).tobytes()
    ranks = [np.load(os.path.join(tmp_path, "resume%d.npz" % r)) for r in range(4)]
    for d in ranks:
        assert d["loaded"].tobytes() == saved.tobytes()
    full = z.consolidate_state([torch.load(os.path.join(tmp_path, "ckpt%d.pt" % r))
                                for r in range(2)])
    numel = full["numel"]
    S = oracle.shard_size(numel, 4)
    P = 4 * S
    x, m, v = (np.zeros(P, np.float32) for _ in range(3))
    x[:numel], m[:numel], v[:numel] = (full[k].numpy() for k in ("master", "m", "v"))
    params = np.zeros(P, np.float32)
    t = full["t"]
    assert t == 2
    for j in range(2):
        g = [np.ascontiguousarray(d["grads"][j], np.float32) for d in ranks]
        oracle.zero_step(g, oracle.F32, numel, x, m, v, params, oracle.F32, LR, 0.9, 0.999,
                         1e-8, t + 1)
        t += 1
    for r, d in enumerate(ranks):
        assert int(d["t"]) == 4
        assert d["final"].tobytes() == params[:numel].tobytes(), r
        assert d["master"].tobytes() == x[r * S:(r + 1) * S].tobytes(), r
