"""bench.py on CPU: the reference arm in one process and under two torchrun
ranks over gloo (rank 0 alone prints one JSON line; the other rank exits 0
without work), and the oracle timing split over host threads."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(cmd):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    return lines


def _check(line):
    d = json.loads(line)
    assert d["impl"] == "reference" and d["unit"] == "params/s" and d["value"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["higher_is_better"] is True
    return d


def test_reference_arm_single_process():
    lines = _run([sys.executable, "bench.py", "--impl", "reference", "--workload", "gpt2_small",
                  "--steps", "1", "--warmup", "1"])
    assert len(lines) == 1
    _check(lines[0])


def test_threaded_oracle_timing_steps_independent_pieces():
    """The all-cores timing steps contiguous pieces of the sample on separate
    threads.  That measures the same work as one thread only because the
    update is elementwise: stepping the pieces gives, element for element,
    what one call on the whole sample gives."""
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    import oracle
    import workloads as W
    w = W.gpt2_xl()                       # 16 fp16 ranks, loss-scaled
    n = 50_001
    grads, x0 = bench.oracle_sample(w, n)

    def run(lo, hi):
        k = hi - lo
        P = oracle.shard_size(k, w.world) * w.world
        x = np.zeros(P, np.float32)
        x[:k] = x0[lo:hi]
        m, v = np.zeros(P, np.float32), np.zeros(P, np.float32)
        out = np.zeros(P, oracle.NP_STORAGE[w.param_dtype])
        for t in (1, 2):
            oracle.zero_step([g[lo:hi] for g in grads], w.grad_dtype, k, x, m, v, out,
                             w.param_dtype, w.lr, w.beta1, w.beta2, w.eps, t,
                             loss_scale=w.loss_scale)
        return x[:k], m[:k], v[:k], out[:k]

    whole = run(0, n)
    cuts = [0, 7, 20_000, 33_333, n]
    for a, b in zip(cuts, cuts[1:]):
        for got, want in zip(run(a, b), whole):
            assert got.tobytes() == want[a:b].tobytes()
    # and the threaded timing runs on both views
    n_s, times = bench.oracle_time(W.gpt2_small(), 1 << 16, 2, threads=4)
    assert n_s == 1 << 16 and len(times) == 2 and all(t > 0 for t in times)
    n_s, times = bench.oracle_time(W.one_rank_7p5b(0), 1 << 15, 1, threads=3)
    assert n_s == 1 << 15 and len(times) == 1


def test_reference_arm_under_torchrun_two_ranks():
    lines = _run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                  "--nproc-per-node", "2", "--master-addr", "127.0.0.1", "--master-port", "29531",
                  "bench.py", "--impl", "reference", "--workload", "gpt2_small", "--gpus", "2",
                  "--steps", "1", "--warmup", "1"])
    assert len(lines) == 1
    d = _check(lines[0])
    assert d["n_gpus"] == 2 and d["scaling"] == "strong"
    # the config the GPU arm's sharded mode prints for the same launch
    sys.path.insert(0, ROOT)
    import bench
    old = sys.argv
    sys.argv = ["bench.py", "--workload", "gpt2_small", "--gpus", "2"]
    try:
        args = bench.parse()
    finally:
        sys.argv = old
    args.dist_backend = "gloo"
    assert d["config"] == bench.sharded_config(args, 2)


def _plan_bytes(w, shadow=False):
    """The bench's per-step algorithmic bytes for a workload, from its launch
    plan built on a stand-in for the GPU runner (no launch is made)."""
    sys.path.insert(0, ROOT)
    import bench
    return bench.static_plan_bytes(w, shadow)


def test_reference_arm_prints_the_gpu_arms_config():
    """Both arms describe the run with the same `config` dictionary: the
    default command line (GPT-2 XL headline plus the four other workloads)
    and a single-workload one."""
    sys.path.insert(0, ROOT)
    import bench
    for extra in ([], ["--workload", "gpt2_small"]):
        lines = _run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                      "--warmup", "1", *extra])
        d = _check(lines[0])
        old = sys.argv
        sys.argv = ["bench.py", *extra]
        try:
            want = bench.static_config(bench.parse(), 1)
        finally:
            sys.argv = old
        assert d["config"] == want
        assert ("workloads" in want) == (not extra)
    assert set(want) >= {"workload", "params_updated_per_step", "alg_bytes_per_step"}


def test_algorithmic_bytes_match_the_closed_forms():
    """The bytes behind every roofline figure: per parameter N*b_g + 24 + b_p
    for the fused step (+ b_g with the all-reduce output), 36 + 30 for the
    two passes, 2*b_p per placed element, two unit gathers per ZeRO-3 step."""
    sys.path.insert(0, ROOT)
    import workloads as W
    xl = W.gpt2_xl()
    psi = xl.numel
    assert _plan_bytes(xl, shadow=True) == 58 * psi == 90_341_449_600
    assert _plan_bytes(xl) == (16 * 2 + 4) * psi + (4 + 24 + 2) * psi        # two passes
    assert _plan_bytes(W.gpt2_xl_adamw(), shadow=True) == 58 * psi
    assert _plan_bytes(W.gpt2_xl_bucketed(), shadow=True) == 58 * psi
    # bucketed, loss-scaled with one state set: a reduce per bucket, one apply
    assert _plan_bytes(W.gpt2_xl_bucketed()) == (16 * 2 + 4) * psi + (4 + 24 + 2) * psi
    # bucketed without loss scaling: the buckets' fused passes only
    assert _plan_bytes(W.gpt2_xl_bucketed().replace(loss_scale=0.0)) == 58 * psi
    sm = W.gpt2_small()
    assert _plan_bytes(sm) == 42 * sm.numel
    assert _plan_bytes(W.gpt2_small_stage1()) == 44 * sm.numel
    one = W.one_rank_7p5b(0)
    S = one.shard
    assert _plan_bytes(one) == (64 * 2 + 26) * S + 63 * 2 * 2 * S == 47_578_125_000
    z3 = W.zero3_llama7b()
    Su = z3.unit_shard(0)
    assert _plan_bytes(z3) == 32 * (2 * 2 * 2 * 8 + 8 * 2 + 26) * Su == 85_810_544_640
    f16 = W.zero3_llama7b_fp16()
    assert _plan_bytes(f16, shadow=True) == 32 * (2 * 2 * 2 * 8 + 8 * 2 + 26) * Su
    assert _plan_bytes(f16) == 32 * (2 * 2 * 2 * 8 + (8 * 2 + 4) + (4 + 24 + 2)) * Su
    fs = W.fsdp2_llama7b()
    assert sum(fs.unit_shard(u) for u in range(len(fs.units))) == 32 * Su
    assert _plan_bytes(fs) == _plan_bytes(W.fsdp2_llama7b_per_param()) == 85_810_544_640


def test_forward_runs_pair_only_small_units():
    """The ZeRO-3 forward's gather calls: consecutive units whose shards are
    both under 32 MiB go in pairs, larger ones alone, an odd one out last;
    every unit exactly once, in order."""
    sys.path.insert(0, ROOT)
    import workloads as W
    from workloads.runner import forward_runs
    assert forward_runs(W.zero3_gpt2_small()) == [(u, 2) for u in range(0, 14, 2)]
    assert forward_runs(W.zero3_llama7b(4)) == [(u, 1) for u in range(4)]
    assert forward_runs(W.zero3_gpt2_small(), pairs=False) == [(u, 1) for u in range(14)]
    # 8 ranks of bf16: 134,217,728 elements make a 32 MiB shard
    big = 8 * (16 << 20)
    w = W.Workload("mix", 0, 8, 3, W.BF16, W.BF16, rank=0,
                   units=[1000, 2000, big, 3000, 4000, 5000, big - 8, 7])
    w = w.replace(numel=sum(w.units))
    runs = forward_runs(w)
    assert runs == [(0, 2), (2, 1), (3, 2), (5, 2), (7, 1)]
    covered = [u for f, n in runs for u in range(f, f + n)]
    assert covered == list(range(len(w.units)))


def test_backward_chunks_of_small_units():
    """The ZeRO-3 backward in chunks of two from the last unit down (an odd
    one out at unit 0) when every unit is small; none when any shard is 32
    MiB or more, or with pairs off."""
    sys.path.insert(0, ROOT)
    import workloads as W
    from workloads.runner import backward_chunks
    assert backward_chunks(W.zero3_gpt2_small()) == [(u, 2) for u in range(12, -1, -2)]
    assert backward_chunks(W.zero3_llama7b(4)) is None
    assert backward_chunks(W.zero3_gpt2_small(), pairs=False) is None
    w = W.Workload("odd", 0, 4, 3, W.BF16, W.BF16, rank=0, units=[10, 20, 30, 40, 50])
    w = w.replace(numel=sum(w.units))
    chunks = backward_chunks(w)
    assert chunks == [(3, 2), (1, 2), (0, 1)]
    covered = [u for f, n in chunks for u in reversed(range(f, f + n))]
    assert covered == [4, 3, 2, 1, 0]
