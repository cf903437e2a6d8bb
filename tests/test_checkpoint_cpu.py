"""Sharded checkpoints across rank counts, on the CPU: consolidate_state and
shard_state move an optimizer state between the whole flat vector and the
shards of any rank count ("PaddlePaddle ZeRO优化": each rank saves and
restores its own shard).  The pins: every shard is the slice [r*S, r*S + S)
of the vector with S = ceil(numel/N) and zeros past numel (the oracle's
layout, oracle.shard_size), and shard -> consolidate returns the vector bit
for bit for every numel and N, padding included."""
import numpy as np
import pytest
import torch

import oracle
import zero_sharded_optimizer_step_gb300 as z


def _full(numel, seed=0):
    g = torch.Generator().manual_seed(seed)
    return {"master": torch.randn(numel, generator=g), "m": torch.randn(numel, generator=g),
            "v": torch.rand(numel, generator=g), "t": 7, "scale": 1024.0, "good_steps": 3,
            "numel": numel}


@pytest.mark.parametrize("numel", [1, 7, 10, 19_210, 100_003])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 7, 16])
def test_shards_are_the_layouts_slices_and_consolidate_back(numel, world):
    full = _full(numel)
    S = oracle.shard_size(numel, world)
    shards = [z.shard_state(full, world, r) for r in range(world)]
    for r, sd in enumerate(shards):
        assert (sd["rank"], sd["world"], sd["numel"], sd["t"]) == (r, world, numel, 7)
        for k in ("master", "m", "v"):
            want = np.zeros(S, np.float32)
            lo, hi = r * S, min(numel, (r + 1) * S)
            if hi > lo:
                want[:hi - lo] = full[k].numpy()[lo:hi]
            assert sd[k].numpy().tobytes() == want.tobytes(), (r, k)
    back = z.consolidate_state(list(reversed(shards)))      # any order
    for k in ("master", "m", "v"):
        assert back[k].numpy().tobytes() == full[k].numpy().tobytes()
    assert (back["t"], back["scale"], back["good_steps"]) == (7, 1024.0, 3)
    # the all-ranks form (ZeroAdam's): N*S elements, the same vector
    one = z.shard_state(full, world)
    assert "rank" not in one and one["master"].numel() == S * world
    assert z.consolidate_state(one)["v"].numpy().tobytes() == full["v"].numpy().tobytes()


def test_reshard_between_rank_counts():
    """4 ranks -> the whole -> 3 ranks -> the whole: nothing lost or moved."""
    full = _full(19_210, seed=1)
    four = [z.shard_state(full, 4, r) for r in range(4)]
    three = [z.shard_state(z.consolidate_state(four), 3, r) for r in range(3)]
    again = z.consolidate_state(three)
    for k in ("master", "m", "v"):
        assert again[k].numpy().tobytes() == full[k].numpy().tobytes()


def test_incomplete_or_inconsistent_checkpoints_are_refused():
    full = _full(1000)
    shards = [z.shard_state(full, 4, r) for r in range(4)]
    with pytest.raises(ValueError):
        z.consolidate_state(shards[:3])                      # a rank missing
    with pytest.raises(ValueError):
        z.consolidate_state(shards[:3] + [shards[0]])        # a rank twice
    bad = dict(shards[2], t=8)
    with pytest.raises(ValueError):
        z.consolidate_state(shards[:2] + [bad, shards[3]])   # the ranks disagree on t
    other = z.shard_state(_full(999), 4, 3)
    with pytest.raises(ValueError):
        z.consolidate_state(shards[:3] + [other])            # another checkpoint's shard
    with pytest.raises(ValueError):
        z.consolidate_state([])
    with pytest.raises(ValueError):
        z.shard_state(full, 4, 4)
