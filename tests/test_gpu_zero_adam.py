"""The ZeroAdam facade (the pages' ZeroAdam(params, lr, betas, eps) with
step, zero_grad and state_bytes) over the C ABI: N ranks' grads written
through per-parameter views, the step bit-identical to the oracle, the
model's parameters updated in place as views of the flat buffer."""
import numpy as np
import pytest
import torch

import oracle
import synth


def _mlp(dt):
    shapes = [(256, 64), (256,), (10, 256), (10,)]
    dev = torch.device("cuda:0")
    out = []
    for i, s in enumerate(shapes):
        n = int(np.prod(s))
        h = synth.fill_host(n, synth.F32, synth.key(11, synth.KIND_MASTER, 0, i), 0.05)
        out.append(torch.from_numpy(h).reshape(s).to(dev, dt))
    return out


@pytest.mark.gpu
@pytest.mark.parametrize("dt,scaled,wd", [(torch.bfloat16, False, 0.0), (torch.float16, True, 0.0),
                                          (torch.float32, False, 0.01)])
def test_zero_adam_matches_the_oracle(dt, scaled, wd):
    import zero_sharded_optimizer_step_gb300 as z
    world, lr, b1, b2, eps = 4, 1e-2, 0.9, 0.999, 1e-8
    params = _mlp(dt)
    opt = z.ZeroAdam(params, world, lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd,
                     loss_scale=2.0 ** 10 if scaled else 0.0)
    code = z.dtype_code(dt)
    numel = opt.numel
    S = oracle.shard_size(numel, world)
    assert opt.state_bytes() == 12 * S
    for p, (off, n) in zip(params, opt._offsets):       # parameters are views of the flat buffer
        assert p.data_ptr() == opt.flat[off:].data_ptr()
    x = opt.master.cpu().numpy().copy()
    m, v = np.zeros_like(x), np.zeros_like(x)
    full = opt.flat.cpu().numpy().copy() if dt == torch.float32 else \
        opt.flat.view(torch.int16).cpu().numpy().view(np.uint16).copy()
    scale, good, t = opt.scale, 0, 0
    skips = []
    for it in (1, 2, 3):
        opt.zero_grad()
        host = []
        for k in range(world):
            g = synth.fill_host(numel, code, synth.key(11, synth.KIND_GRAD, it, k),
                                1e-3 * (scale if scaled else 1.0))
            if scaled and it == 2 and k == 1:
                g[123] = oracle.cast(np.array([np.inf], np.float32), code)[0]
            host.append(g)
            flat = torch.from_numpy(g.view(np.int16) if code else g).to("cuda:0")
            flat = flat.view(dt) if code else flat
            off = 0
            for view in opt.rank_grads(k):               # a backward writing per parameter
                view.copy_(flat[off:off + view.numel()].view_as(view))
                off += view.numel()
        skipped = opt.step()
        sk, _ = oracle.zero_step(host, code, numel, x, m, v, full, code, lr, b1, b2, eps, t + 1,
                                 loss_scale=scale if scaled else 0.0, weight_decay=wd)
        assert skipped == sk
        skips.append(sk)
        if not sk:
            t += 1
        if scaled:
            scale, good = oracle.scale_update(scale, sk, good, 2000)
    torch.cuda.synchronize()
    if scaled:
        assert skips == [False, True, False] and opt.scale == scale == 2.0 ** 9
    assert opt.t == t
    gx, gm, gv = (a.cpu().numpy() for a in opt.state())
    assert gx.tobytes() == x.tobytes() and gm.tobytes() == m.tobytes() and gv.tobytes() == v.tobytes()
    got = opt.flat.cpu().numpy() if dt == torch.float32 else \
        opt.flat.view(torch.int16).cpu().numpy().view(np.uint16)
    assert got.tobytes() == full.tobytes()
    # the model's parameters see the update
    off = 0
    for p in params:
        assert torch.equal(p.reshape(-1), opt.flat[off:off + p.numel()])
        off += p.numel()
    opt.close()


@pytest.mark.gpu
def test_zero_adam_trains_the_pages_mlp_like_torch_adam():
    """The pages' check ("ZeRO 与 FSDP…", 从零实现 ZeRO 的 Adam): the MLP
    Linear(64,256)+GELU+Linear(256,10) trained by 4 data-parallel ranks with
    equal local batches through ZeroAdam ends where single-process
    torch.optim.Adam on the full batch ends, within the pages' 1e-5.  The
    ranks' backward passes run through torch autograd on this GPU; each
    writes its local grads into its rank's views."""
    import copy
    import zero_sharded_optimizer_step_gb300 as z
    torch.manual_seed(0)
    dev = torch.device("cuda:0")
    model = torch.nn.Sequential(torch.nn.Linear(64, 256), torch.nn.GELU(),
                                torch.nn.Linear(256, 10)).to(dev)
    ref = copy.deepcopy(model)
    world, per_rank, lr = 4, 8, 1e-2
    opt = z.ZeroAdam(list(model.parameters()), world, lr=lr, betas=(0.9, 0.999), eps=1e-8)
    ref_opt = torch.optim.Adam(ref.parameters(), lr=lr, betas=(0.9, 0.999), eps=1e-8)
    assert opt.numel == 19_210
    assert opt.state_bytes() == 57_636          # the pages' printed per-rank figure
    loss_fn = torch.nn.CrossEntropyLoss()
    for it in range(5):
        x = torch.randn(world * per_rank, 64, device=dev)
        y = torch.randint(0, 10, (world * per_rank,), device=dev)
        opt.zero_grad()
        for k in range(world):
            model.zero_grad(set_to_none=True)
            sl = slice(k * per_rank, (k + 1) * per_rank)
            loss_fn(model(x[sl]), y[sl]).backward()
            for view, p in zip(opt.rank_grads(k), model.parameters()):
                view.copy_(p.grad)
        assert opt.step() is False
        ref_opt.zero_grad(set_to_none=True)
        loss_fn(ref(x), y).backward()
        ref_opt.step()
    torch.cuda.synchronize()
    worst = max((a - b).abs().max().item() for a, b in zip(model.parameters(), ref.parameters()))
    assert worst < 1e-5, worst
    opt.close()


@pytest.mark.gpu
@pytest.mark.parametrize("dt,scale", [(torch.bfloat16, 0.0), (torch.float16, 2.0 ** 10)])
def test_zero_adam_resumes_from_its_state(dt, scale):
    """Two steps, a checkpoint, two more steps; a fresh model and optimizer
    (other initial weights) loaded from the checkpoint run the same two steps
    to the same bits -- the flat parameters, the state, t and the scale."""
    import zero_sharded_optimizer_step_gb300 as z
    world = 4
    code = z.dtype_code(dt)

    def grads_of(opt, it):
        for k in range(world):
            g = synth.fill_host(opt.numel, code, synth.key(13, synth.KIND_GRAD, it, k),
                                1e-3 * (scale or 1.0))
            flat = torch.from_numpy(g.view(np.int16)).to("cuda:0").view(dt)
            off = 0
            for view in opt.rank_grads(k):
                view.copy_(flat[off:off + view.numel()].view_as(view))
                off += view.numel()

    def run(opt, its):
        for it in its:
            opt.zero_grad()
            grads_of(opt, it)
            opt.step()

    a = z.ZeroAdam(_mlp(dt), world, lr=1e-2, loss_scale=scale)
    run(a, [1, 2])
    sd = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in a.state_dict().items()}
    run(a, [3, 4])
    b = z.ZeroAdam([p * 0 + 0.5 for p in _mlp(dt)], world, lr=1e-2, loss_scale=scale)
    b.load_state_dict(sd)
    run(b, [3, 4])
    torch.cuda.synchronize()
    assert torch.equal(a.flat, b.flat)
    for x, y in zip(a.state(), b.state()):
        assert torch.equal(x, y)
    assert a.t == b.t == 4 and a.scale == b.scale
    a.close()
    b.close()
