"""The seeded input generator: C host fill == numpy restatement, moments of
the draws, bounded range (what makes the overflow pattern of the loss-scaled
workload a property of its construction)."""
import numpy as np
import pytest

import synth


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16, synth.F16])
def test_host_fill_matches_numpy(dtype):
    for seed, kind, step, rank, unit in [(0, 1, 1, 0, 0), (7, 1, 3, 5, 0), (0, 0, 0, 0, 31)]:
        k = synth.key(seed, kind, step, rank, unit)
        assert k == synth.py_key(seed, kind, step, rank, unit)
        a = synth.fill_host(50000, dtype, k, 0.065536, index0=(1 << 33) + 17)
        b = synth.np_fill(50000, dtype, k, 0.065536, index0=(1 << 33) + 17)
        assert a.tobytes() == b.tobytes()
        idx = np.array([0, 5, 3, 1 << 40, 99], np.int64)
        c = synth.fill_host(5, dtype, k, 0.01, indices=idx)
        d = synth.np_fill(5, dtype, k, 0.01, indices=idx)
        assert c.tobytes() == d.tobytes()
        # random access equals the contiguous fill at the same positions
        e = synth.fill_host(100, dtype, k, 0.01)
        f = synth.fill_host(3, dtype, k, 0.01, indices=np.array([0, 50, 99]))
        assert f.tobytes() == e[[0, 50, 99]].tobytes()


def test_moments_and_range():
    k = synth.key(3, synth.KIND_GRAD, 1, 0)
    x = synth.fill_host(1 << 21, synth.F32, k, 1e-3).astype(np.float64)
    assert abs(x.mean()) < 3e-6
    assert abs(x.std() / 1e-3 - 1) < 3e-3
    # |c| <= 131070, so |x| <= 131070 * sigma / 37837.2... ~ 3.4641 sigma
    assert np.abs(x).max() <= 131070 / synth.IH_STD * 1e-3 * (1 + 1e-6)
    # 4th moment of the Irwin-Hall(4) shape: kurtosis 3 - 6/(5*4) = 2.7
    kurt = ((x - x.mean()) ** 4).mean() / x.var() ** 2
    assert abs(kurt - 2.7) < 0.02


def test_streams_are_distinct():
    a = synth.fill_host(1000, synth.F32, synth.key(0, 1, 1, 0), 1.0)
    b = synth.fill_host(1000, synth.F32, synth.key(0, 1, 1, 1), 1.0)
    c = synth.fill_host(1000, synth.F32, synth.key(0, 1, 2, 0), 1.0)
    d = synth.fill_host(1000, synth.F32, synth.key(1, 1, 1, 0), 1.0)
    for u, w in [(a, b), (a, c), (a, d), (b, c)]:
        assert abs(np.corrcoef(u, w)[0, 1]) < 0.15


def test_pick_index_in_range():
    for n in (1, 7, 1_557_611_200):
        i = synth.pick_index(0, n, step=3, rank=5)
        assert 0 <= i < n
