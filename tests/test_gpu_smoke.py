"""The build entry's smoke() (one small step sequence on cuda:0 through the
C ABI, checked against the oracle) stays green with the rest of the GPU
tests."""
import pytest


@pytest.mark.gpu
def test_smoke_entry_point():
    import __graft_entry__
    __graft_entry__.smoke()
