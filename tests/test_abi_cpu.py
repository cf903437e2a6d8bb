"""The C ABI without a GPU: the library builds and loads, exports every
function include/zero.h declares, and its host-only logic (geometry, closed
forms, loss-scale policy, argument checks) behaves."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "zero.h")


@pytest.fixture(scope="module")
def z():
    import __graft_entry__
    __graft_entry__._library_builder().build()
    import zero_sharded_optimizer_step_gb300 as z
    return z


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[a-z_][\w\s\*]*?\b(zero\w*)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ["zero_init", "zero_bind", "zero_step", "zero_step_reduce", "zero_step_apply",
                 "zero_step_status", "zero_allgather", "zero3_gather_unit", "zero3_step_unit",
                 "zero3_reduce_unit", "zero_state_bytes", "zero_model_state_bytes",
                 "zero_destroy", "zero_strerror", "zero_shard_size"]:
        assert must in names


def test_library_exports_every_declared_symbol(z):
    lib = ctypes.CDLL(z.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    out = subprocess.run(["nm", "-D", "--defined-only", z.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (zero\w*)$", out, flags=re.M))
    assert set(declared_functions()) <= exported
    # the binding wraps exactly the declared entry points
    assert set(z.EXPORTED) == set(declared_functions())


def test_header_compiles_as_c():
    src = '#include "zero.h"\nint main(void){return ZERO_OK;}\n'
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER),
                    "-x", "c", "-", "-o", os.devnull], input=src, text=True, check=True)


def test_error_codes_match_the_header(z):
    """The binding's codes equal the header's enum, and every code has its
    own message (no GPU needed)."""
    text = open(HEADER).read()
    import re
    enum = dict((k, int(v)) for k, v in re.findall(r"(ZERO_[A-Z]+) = (-?\d+)", text)
                if k in ("ZERO_OK", "ZERO_SKIPPED", "ZERO_EINVAL", "ZERO_ECUDA", "ZERO_EALIGN",
                         "ZERO_ESTATE", "ZERO_ETIMEOUT"))
    assert len(enum) == 7
    msgs = set()
    for name, code in enum.items():
        assert getattr(z, name) == code
        msg = z.zero_strerror(code)
        assert msg.startswith(name)
        msgs.add(msg)
    assert len(msgs) == 7 and z.zero_strerror(-99) == "unknown zero code"


def test_host_geometry_and_closed_forms(z):
    import oracle
    from oracle import memory as mem
    for numel in (0, 1, 5, 19210, 7_500_000_000, 1_557_611_200):
        for n in (1, 3, 4, 16, 64, 256):
            assert z.zero_shard_size(numel, n) == oracle.shard_size(numel, n)
    assert z.zero_shard_size(5, 0) == -1
    for stage in range(4):
        for psi, n in [(7 * 10**9, 8), (13 * 10**9, 16), (7_500_000_000, 64)]:
            got = z.zero_model_state_bytes(psi, n, stage)
            want = float(mem.model_state_bytes(psi, n, stage))
            assert got == pytest.approx(want, rel=1e-15)
    assert z.zero_model_state_bytes(1, 1, 4) == -1.0


def test_scale_update_matches_oracle(z):
    import oracle
    s_z, g_z = 65536.0, 0
    s_o, g_o = 65536.0, 0
    pattern = [False] * 5 + [True] + [False] * 12 + [True, True] + [False] * 30
    for sk in pattern:
        s_z, g_z = z.zero_scale_update(s_z, sk, g_z, 10)
        s_o, g_o = oracle.scale_update(s_o, sk, g_o, 10)
        assert (s_z, g_z) == (s_o, g_o)


def test_init_validation(z):
    bad = [
        dict(numel=10, world=0, stage=2),
        dict(numel=10, world=257, stage=2),
        dict(numel=10, world=4, stage=0),
        dict(numel=10, world=4, stage=4),
        dict(numel=-1, world=4, stage=2),
        dict(numel=10, world=4, stage=2, rank=4),
        dict(numel=10, world=4, stage=2, rank=-2),
        dict(numel=10, world=4, stage=2, grad_dtype=7),
        dict(numel=10, world=4, stage=2, unit_numels=[5, 5]),
        dict(numel=10, world=4, stage=3),
        dict(numel=11, world=4, stage=3, unit_numels=[5, 5]),
        dict(numel=10, world=4, stage=3, unit_numels=[5, -5, 10]),
    ]
    for kw in bad:
        args = dict(grad_dtype=z.ZERO_BF16, param_dtype=z.ZERO_BF16, rank=-1, unit_numels=None)
        args.update(kw)
        with pytest.raises(z.ZeroError) as ei:
            z.zero_init(args["numel"], args["world"], args["stage"], args["grad_dtype"],
                        args["param_dtype"], args["rank"], args["unit_numels"])
        assert ei.value.code == z.ZERO_EINVAL
        assert z.zero_last_error()


def test_view_of_several_ranks(z):
    """zero_init_ranks: ranks [r, r + k) of N; the state is their k shards
    end to end (per unit for stage 3), the parameter buffer the whole vector
    (stages 1 and 2) or the view's persistent shards (stage 3)."""
    c = z.zero_init_ranks(19210, 4, 2, z.ZERO_F32, z.ZERO_F32, 1, 3)
    assert z.zero_ctx_shard_size(c, -1) == 4803
    assert z.zero_ctx_state_elems(c) == 3 * 4803
    assert z.zero_ctx_param_elems(c) == 19212
    assert z.zero_state_bytes(c) == 3 * 57636
    # k = 1 is one rank's view; ranks 0..N-1 the all-ranks view's state
    assert z.zero_ctx_state_elems(z.zero_init_ranks(19210, 4, 1, z.ZERO_F32, z.ZERO_F32, 3,
                                                    1)) == 4803
    assert z.zero_ctx_state_elems(z.zero_init_ranks(19210, 4, 2, z.ZERO_F32, z.ZERO_F32, 0,
                                                    4)) == 19212
    for first, k, stage in ((0, 0, 2), (-1, 2, 2), (2, 3, 2), (4, 1, 2), (0, 2, 0)):
        with pytest.raises(z.ZeroError) as ei:
            z.zero_init_ranks(19210, 4, stage, z.ZERO_F32, z.ZERO_F32, first, k)
        assert ei.value.code == z.ZERO_EINVAL, (first, k, stage)
        assert z.zero_last_error()
    # stage 3: per unit the view's k shards end to end; units are required
    with pytest.raises(z.ZeroError):
        z.zero_init_ranks(19210, 4, 3, z.ZERO_F32, z.ZERO_F32, 0, 2)
    units = [10, 7, 33]                       # S_u = 3, 2, 9 over 4 ranks
    c3 = z.zero_init_ranks(sum(units), 4, 3, z.ZERO_BF16, z.ZERO_BF16, 1, 2, units)
    assert [z.zero_ctx_shard_size(c3, u) for u in range(3)] == [3, 2, 9]
    assert [z.zero_ctx_unit_state_offset(c3, u) for u in range(3)] == [0, 6, 10]
    assert z.zero_ctx_state_elems(c3) == 28 and z.zero_ctx_param_elems(c3) == 28


def test_context_geometry(z):
    c = z.zero_init(19210, 4, 2, z.ZERO_F32, z.ZERO_F32, -1)
    assert z.zero_ctx_shard_size(c, -1) == 4803
    assert z.zero_ctx_state_elems(c) == 19212
    assert z.zero_ctx_param_elems(c) == 19212
    c1 = z.zero_init(19210, 4, 2, z.ZERO_F32, z.ZERO_F32, 2)
    assert z.zero_ctx_state_elems(c1) == 4803
    assert z.zero_state_bytes(c1) == 57636          # ZeroAdam.state_bytes() per rank
    units = [10, 7, 33]
    c3 = z.zero_init(sum(units), 4, 3, z.ZERO_BF16, z.ZERO_BF16, 1, units)
    S = [3, 2, 9]
    assert [z.zero_ctx_shard_size(c3, u) for u in range(3)] == S
    assert [z.zero_ctx_unit_state_offset(c3, u) for u in range(3)] == [0, 3, 5]
    assert z.zero_ctx_state_elems(c3) == 14 and z.zero_ctx_param_elems(c3) == 14
    c3a = z.zero_init(sum(units), 4, 3, z.ZERO_BF16, z.ZERO_BF16, -1, units)
    assert [z.zero_ctx_unit_param_offset(c3a, u) for u in range(3)] == [0, 12, 20]
    assert z.zero_ctx_state_elems(c3a) == 56
    assert z.zero_ctx_shard_size(c3a, 3) == -1 and z.zero_ctx_shard_size(c3a, -1) == -1
    c0 = z.zero_init(0, 8, 2, z.ZERO_BF16, z.ZERO_BF16, -1)
    assert z.zero_ctx_state_elems(c0) == 0


def test_calls_before_bind_fail_cleanly(z):
    c = z.zero_init(100, 4, 2, z.ZERO_BF16, z.ZERO_BF16, -1)
    with pytest.raises(z.ZeroError) as ei:
        z.zero_step(c, [0, 0, 0, 0], 1e-3, 0.9, 0.999, 1e-8, 1, stream=0)
    assert ei.value.code == z.ZERO_ESTATE
    with pytest.raises(z.ZeroError) as ei:
        z.zero_step_status(c)
    assert ei.value.code == z.ZERO_ESTATE
    with pytest.raises(z.ZeroError):
        z.zero3_begin_step(c)   # not stage 3


def test_step_occupancy_argument_checked(z):
    c = z.zero_init(1000, 4, 2, z.ZERO_BF16, z.ZERO_BF16, -1)
    for ok in (0, 1, 4, 32):
        z.zero_set_step_occupancy(c, ok)
    for bad in (-1, 33):
        with pytest.raises(z.ZeroError) as ei:
            z.zero_set_step_occupancy(c, bad)
        assert ei.value.code == z.ZERO_EINVAL


def test_advance_state_rejects_a_non_finite_scale(z):
    buf = np.zeros(z.ZERO_ADVANCE_STATE_BYTES, np.uint8)
    for bad in (float("inf"), float("nan")):
        with pytest.raises(z.ZeroError) as ei:
            z.zero_advance_state(buf.ctypes.data, 1, bad, 2000)
        assert ei.value.code == z.ZERO_EINVAL


def test_advance_table_and_state_on_the_host(z):
    """The device-advance table holds, per step, the bias corrections the
    oracle derives for that step (bit for bit), and the state block packs t,
    scale, status, good steps and the growth interval in 32 bytes."""
    import oracle
    T = 3000
    buf = np.zeros(z.zero_advance_table_bytes(T) // 4, np.float32)
    assert buf.size == 2 * T
    z.zero_fill_advance_table(buf.ctypes.data, T, 0.9, 0.999)
    for t in (1, 2, 3, 17, 100, 999, 3000):
        sc = oracle.adam_scalars(0.9, 0.999, t)       # c1, c2, bc1, bc2
        assert buf[2 * (t - 1)].tobytes() == sc[2].tobytes()
        assert buf[2 * (t - 1) + 1].tobytes() == sc[3].tobytes()
    assert z.zero_advance_table_bytes(0) == -1
    st = np.zeros(4, np.int64)
    z.zero_advance_state(st.ctypes.data, 7, 65536.0, 2000)
    assert st[0] == 7 and st[2] == 0 and st[3] == 2000
    assert np.frombuffer(st[1].tobytes()[:4], np.float32)[0] == 65536.0
    assert np.frombuffer(st[1].tobytes()[4:], np.int32)[0] == 0
    with pytest.raises(z.ZeroError):
        z.zero_fill_advance_table(None, 5, 0.9, 0.999)
