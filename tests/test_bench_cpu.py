"""bench.py's reference arm on CPU: one process and two torchrun ranks over
gloo (rank 0 alone prints one JSON line; the other rank exits 0 without
work)."""
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
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["higher_is_better"] is True
    return d


def test_reference_arm_single_process():
    lines = _run([sys.executable, "bench.py", "--impl", "reference", "--workload", "gpt2_small",
                  "--steps", "1", "--warmup", "1"])
    assert len(lines) == 1
    _check(lines[0])


def test_reference_arm_under_torchrun_two_ranks():
    lines = _run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                  "--nproc-per-node", "2", "--master-addr", "127.0.0.1", "--master-port", "29531",
                  "bench.py", "--impl", "reference", "--workload", "gpt2_small", "--gpus", "2",
                  "--steps", "1", "--warmup", "1"])
    assert len(lines) == 1
    assert _check(lines[0])["n_gpus"] == 2
