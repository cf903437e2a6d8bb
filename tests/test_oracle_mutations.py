"""The pins catch plausible mistakes in the oracle.  Each case plants one
mistake in a copy of oracle/zero_oracle.c (on the CPU), builds it, and runs
the oracle's pin tests against that copy: at least one pin must fail."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "zero_oracle.c")
PIN_TESTS = ["tests/test_oracle_adam.py", "tests/test_oracle_layout.py",
             "tests/test_oracle_cast_skip.py", "tests/test_oracle_dim0.py"]

MUTANTS = [
    ("weight of g in m dropped", "out[0] = (float)(1.0 - beta1);", "out[0] = (float)(1.0);"),
    ("bias correction at t+1", "out[2] = (float)(1.0 - pow(beta1, (double)t));",
     "out[2] = (float)(1.0 - pow(beta1, (double)(t + 1)));"),
    ("v from g, not g*g", "float vj = v[j] * b2 + c2 * (gj * gj);",
     "float vj = v[j] * b2 + c2 * gj;"),
    ("eps inside the root", "float den = sqrtf(vh) + epsf;", "float den = sqrtf(vh + epsf);"),
    ("update added", "x[j] = xj - upd;", "x[j] = xj + upd;"),
    ("betas swapped in m", "float mj = m[j] * b1 + c1 * gj;", "float mj = m[j] * b2 + c2 * gj;"),
    ("no average over ranks", "float x = acc[j] / w;", "float x = acc[j];"),
    ("no unscale", "if (loss_scale > 0.0f) x = x / loss_scale;", ";"),
    ("floor shard size", "return (numel + world - 1) / world;", "return numel / world;"),
    ("bf16 truncates", "if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) hi += 1u;", ";"),
    ("shards placed one slot late", "memcpy((char *)full + ((int64_t)r * S + j) * es,",
     "memcpy((char *)full + ((int64_t)((r + 1) % world) * S + j) * es,"),
    ("overflow never skips", "if (loss_scale > 0.0f && bad > 0) return 1;", "if (0) return 1;"),
    ("overflow tested before the unscale",
     "        if (loss_scale > 0.0f) x = x / loss_scale;\n        g[j] = x;\n"
     "        if (!isfinite(x)) ++bad;",
     "        if (!isfinite(x)) ++bad;\n        if (loss_scale > 0.0f) x = x / loss_scale;\n"
     "        g[j] = x;"),
    ("last rank left out of the sum",
     "for (int32_t k = 1; k < world; ++k) a = a + widen(grads[k], dtype, i);",
     "for (int32_t k = 1; k < world - 1; ++k) a = a + widen(grads[k], dtype, i);"),
    ("padding reads a real grad", "if (j >= n_valid) { acc[j] = 0.0f; continue; }",
     "if (j > n_valid) { acc[j] = 0.0f; continue; }"),
    ("decay without lr", "const float decay = (float)(1.0 - lr * weight_decay);",
     "const float decay = (float)(1.0 - weight_decay);"),
    ("dim-0 shard not whole rows", "return (rows + world - 1) / world * row_elems;",
     "return (rows * row_elems + world - 1) / world;"),
    ("scale doubled on a skip", "return scale * 0.5f;", "return scale * 2.0f;"),
    ("scale grows to infinity", "return isfinite(grown) ? grown : scale;", "return grown;"),
    ("scale grows by 4", "const float grown = scale * 2.0f;", "const float grown = scale * 4.0f;"),
    ("clean-step count kept after growth",
     "        *good_steps = 0;\n        /* grow only to a finite scale */",
     "        /* grow only to a finite scale */"),
]


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, source, name, old, new):
    assert source.count(old) >= 1, "the mutation no longer applies: " + name
    mutant = tmp_path / "mutant.c"
    mutant.write_text(source.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-std=c11", "-fPIC", "-shared", "-o",
                    str(lib), str(mutant), "-lm"], check=True)
    env = dict(os.environ, ZERO_ORACLE_LIB=str(lib))
    out = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                          *PIN_TESTS], cwd=ROOT, env=env, capture_output=True, text=True,
                         timeout=600)
    assert out.returncode != 0, "no pin caught: " + name


def test_unmutated_copy_passes(tmp_path, source):
    """The harness itself: an unchanged copy passes every pin."""
    lib = tmp_path / "libsame.so"
    src = tmp_path / "same.c"
    src.write_text(source)
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-std=c11", "-fPIC", "-shared", "-o",
                    str(lib), str(src), "-lm"], check=True)
    env = dict(os.environ, ZERO_ORACLE_LIB=str(lib))
    out = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                          *PIN_TESTS], cwd=ROOT, env=env, capture_output=True, text=True,
                         timeout=600)
    assert out.returncode == 0, out.stdout[-2000:]
