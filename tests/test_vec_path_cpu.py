"""The step kernels' choice between the vector path and the per-element
path, checked on the CPU: zgb::step_vector_path_ok, the one predicate every
launch (zero_step_noalloc included) takes its vec_ok from, and
zgb::step_grad_align, the width the vector path reads the rank grads with,
compiled from the library's internal header into a small host program.

An fp32 buffer the vector path would touch at an address off a 16-byte
boundary, or a grad buffer off an 8-byte one, must send the launch down the
per-element path; that is what keeps a misaligned second state set,
scratch or grad buffer from a misaligned vector access on the GPU.  Grads
on an 8-byte boundary are read 8 bytes per load."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "zero_sharded_optimizer_step_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <cstring>
#include "zero_internal.h"

static char pool[1 << 12] __attribute__((aligned(256)));

static float *f(int byte_off) { return reinterpret_cast<float *>(pool + 256 + byte_off); }

static zgb::StepArgs base(int world)
{
    zgb::StepArgs a;
    memset(&a, 0, sizeof a);
    a.world = world;
    a.master = f(0); a.m = f(64); a.v = f(128); a.g = nullptr;
    for (int k = 0; k < world; ++k) a.grads[k] = f(192 + 32 * k);
    return a;
}

int main()
{
    int fails = 0;
#define EXPECT(cond, want) do { bool got = (cond); if (got != (want)) { \
        printf("FAIL %s: got %d\n", #cond, (int)got); ++fails; } } while (0)
    zgb::StepArgs a = base(4);
    EXPECT(zgb::step_vector_path_ok(a), true);
    // each buffer of the vector path, 4 bytes off
    a = base(4); a.master = f(4);           EXPECT(zgb::step_vector_path_ok(a), false);
    a = base(4); a.m = f(68);               EXPECT(zgb::step_vector_path_ok(a), false);
    a = base(4); a.v = f(132);              EXPECT(zgb::step_vector_path_ok(a), false);
    a = base(4); a.g = f(900);              EXPECT(zgb::step_vector_path_ok(a), false);
    a = base(4); a.g = f(896);              EXPECT(zgb::step_vector_path_ok(a), true);
    a = base(4); a.grads[3] = f(292);       EXPECT(zgb::step_vector_path_ok(a), false);
    // grads on an 8-byte boundary (a rank's slice of a flat vector whose
    // shard length is 4 mod 8 elements) keep the vector path, read in halves
    a = base(4);                            EXPECT(zgb::step_grad_align(a) == 16, true);
    a = base(4); a.grads[1] = f(232);       EXPECT(zgb::step_vector_path_ok(a), true);
                                            EXPECT(zgb::step_grad_align(a) == 8, true);
    a = base(4); a.grads[1] = f(228);       EXPECT(zgb::step_grad_align(a) == 0, true);
    a = base(4); a.grads[0] = f(194);       EXPECT(zgb::step_vector_path_ok(a), false);
    // mixed 16- and 8-byte offsets: the common alignment, 8
    a = base(4); a.grads[2] = f(200);       EXPECT(zgb::step_grad_align(a) == 8, true);
                                            EXPECT(zgb::step_vector_path_ok(a), true);
    // the state stays on 16 bytes: 8 is not enough there
    a = base(4); a.master = f(8);           EXPECT(zgb::step_vector_path_ok(a), false);
    a = base(4); a.grads[2] = nullptr;      EXPECT(zgb::step_vector_path_ok(a), true);
    // a pointer past `world` is never read by the kernels
    a = base(4); a.grads[4] = f(2);         EXPECT(zgb::step_vector_path_ok(a), true);
    // the second state set counts only while it is bound (cur set)
    unsigned long long cur = 0;
    a = base(4); a.xb = f(1024); a.mb = f(1088); a.vb = f(1152); a.cur = &cur;
    EXPECT(zgb::step_vector_path_ok(a), true);
    a.xb = f(1028);                         EXPECT(zgb::step_vector_path_ok(a), false);
    a.xb = f(1024); a.mb = f(1096);         EXPECT(zgb::step_vector_path_ok(a), false);
    a.mb = f(1088); a.vb = f(1156);         EXPECT(zgb::step_vector_path_ok(a), false);
    a.cur = nullptr;                        EXPECT(zgb::step_vector_path_ok(a), true);
    // the params and the stage-1 output are stored at their own alignment
    a = base(4); a.params = pool + 258; a.grad_avg = pool + 262;
    EXPECT(zgb::step_vector_path_ok(a), true);
    // the built-in scratch of zero_step_noalloc is 256-byte aligned; with a
    // 4-byte-aligned second set bound the launch still takes the element path
    a = base(4); a.g = f(1536); a.xb = f(1028); a.mb = f(1088); a.vb = f(1152); a.cur = &cur;
    EXPECT(zgb::step_vector_path_ok(a), false);
    a = base(256);
    for (int k = 0; k < 256; ++k) a.grads[k] = f(0);
    EXPECT(zgb::step_vector_path_ok(a), true);
    a.grads[255] = f(8);                    EXPECT(zgb::step_vector_path_ok(a), true);
                                            EXPECT(zgb::step_grad_align(a) == 8, true);
    a.grads[255] = f(12);                   EXPECT(zgb::step_vector_path_ok(a), false);
    if (fails) return 1;
    printf("ok\n");
    return 0;
}
"""


def _cuda_include():
    for d in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        if d and os.path.exists(os.path.join(d, "include", "cuda_runtime.h")):
            return os.path.join(d, "include")
    return None


def test_vector_path_predicate(tmp_path):
    inc = _cuda_include()
    if inc is None:
        pytest.skip("no CUDA headers")
    src = tmp_path / "vec_path.cpp"
    exe = tmp_path / "vec_path"
    src.write_text(PROGRAM)
    subprocess.run(["g++", "-std=c++17", "-Wall", "-I", CSRC, "-I", inc, str(src), "-o",
                    str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.strip() == "ok"
