"""The library from a plain C program (tests/c_abi_step.c): device memory from
cudaMalloc, the entry points of include/zero.h, no Python or torch in the
process.  On the CPU the program must compile and link against libzero.so;
on a GPU its results -- three loss-scaled steps over two state sets, the
second skipped by a +inf -- must equal the oracle's bit for bit."""
import os
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "zero_sharded_optimizer_step_gb300")
SRC = os.path.join(ROOT, "tests", "c_abi_step.c")
WORLD, NUMEL, SCALES = 3, 100_003, (256.0, 256.0, 128.0)


def _cuda_home():
    for d in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        if d and os.path.exists(os.path.join(d, "include", "cuda_runtime_api.h")):
            return d
    return None


def _build(out_dir):
    import __graft_entry__
    __graft_entry__._library_builder().build()
    cuda = _cuda_home()
    if cuda is None:
        pytest.skip("no CUDA toolkit")
    exe = os.path.join(out_dir, "c_abi_step")
    lib64 = os.path.join(cuda, "lib64")
    subprocess.run(["gcc", "-std=c99", "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(cuda, "include"), SRC, "-o", exe, "-L", PKG, "-lzero",
                    "-L", lib64, "-lcudart", "-Wl,-rpath," + PKG, "-Wl,-rpath," + lib64],
                   check=True)
    return exe


def test_c_program_compiles_and_links(tmp_path):
    exe = _build(str(tmp_path))
    assert os.path.exists(exe)


def _inputs():
    import oracle
    import synth
    x = synth.fill_host(NUMEL, synth.F32, synth.key(9, synth.KIND_MASTER), 0.01)
    grads = []
    for s, scale in enumerate(SCALES):
        step = [synth.fill_host(NUMEL, synth.F16, synth.key(9, synth.KIND_GRAD, s + 1, k),
                                1e-3 * scale) for k in range(WORLD)]
        if s == 1:
            step[2][777] = 0x7C00                 # +inf in fp16: the step is skipped
        grads.append(step)
    return x, grads, oracle


@pytest.mark.gpu
def test_c_program_equals_the_oracle(tmp_path):
    exe = _build(str(tmp_path))
    x0, grads, oracle = _inputs()
    inp, out = os.path.join(tmp_path, "in.bin"), os.path.join(tmp_path, "out.bin")
    with open(inp, "wb") as f:
        f.write(np.int64(NUMEL).tobytes())
        f.write(x0.tobytes())
        for step in grads:
            for g in step:
                f.write(g.tobytes())
    run = subprocess.run([exe, inp, out], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, run.stdout + run.stderr
    S = oracle.shard_size(NUMEL, WORLD)
    P = S * WORLD
    x = np.zeros(P, np.float32)
    x[:NUMEL] = x0
    m, v = np.zeros(P, np.float32), np.zeros(P, np.float32)
    full = np.zeros(P, np.uint16)
    t, skips = 0, []
    for step, scale in zip(grads, SCALES):
        sk, _ = oracle.zero_step(step, oracle.F16, NUMEL, x, m, v, full, oracle.BF16, 1e-3, 0.9,
                                 0.999, 1e-8, t + 1, loss_scale=scale)
        skips.append(int(sk))
        if not sk:
            t += 1
    assert skips == [0, 1, 0]
    got = open(out, "rb").read()
    off = 0
    assert list(np.frombuffer(got[off:off + 12], np.int32)) == skips
    off += 12
    for name, want in (("master", x), ("m", m), ("v", v)):
        assert got[off:off + 4 * P] == want.tobytes(), name
        off += 4 * P
    assert got[off:off + 2 * P] == full.tobytes()
