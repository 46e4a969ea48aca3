"""Pins for the vocabulary-sharded statistics merge (tensor-parallel output layer).

The merge of per-shard statistics must reproduce the statistics of the whole row, which the
oracle's own stats function computes by brute force over all V columns; a hand-worked two-shard
example fixes the arithmetic independently of both."""
import math

import numpy as np
import pytest

import oracle


def _split(V, sizes):
    offs = np.cumsum([0] + list(sizes[:-1]))
    assert sum(sizes) == V
    return offs


def _shard_stats(lg, masked, sizes):
    offs = _split(lg.shape[-1], sizes)
    return [oracle.stats(np.ascontiguousarray(lg[..., o:o + n]), masked)
            for o, n in zip(offs, sizes)], offs


def test_hand_example_two_shards():
    # row [0, ln3 | ln3, 0]: m = ln3, s = 1/3 + 1 + 1 + 1/3 = 8/3, lse = ln 8, conf = 3/8,
    # argmax = 1 (the tie with global id 2 goes to the lower id)
    a, b = oracle.Stats(1), oracle.Stats(1)
    a.row_max[:] = math.log(3); a.lse[:] = math.log(4); a.argmax[:] = 1
    b.row_max[:] = math.log(3); b.lse[:] = math.log(4); b.argmax[:] = 0
    m = oracle.merge_shard_stats([a, b], [0, 2])
    assert m.row_max[0] == math.log(3)
    assert abs(m.lse[0] - math.log(8)) < 1e-15
    assert abs(m.conf[0] - 3 / 8) < 1e-15
    assert m.argmax[0] == 1


@pytest.mark.parametrize("V,sizes", [(10, [5, 5]), (11, [1, 7, 3]), (64, [16] * 4),
                                     (1000, [333, 333, 334]), (37, [1] * 37)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_merge_equals_whole_row(V, sizes, dtype):
    rng = np.random.default_rng(V * 7 + len(sizes))
    x = rng.normal(0, 2, size=(6, V)).astype(np.float32)
    x[0, :] = 0.5                         # every element tied
    x[1, V // 2] = x[1, V - 1] = 9.0      # a tie across shards
    if dtype == "bf16":
        lg = (x.view(np.uint32) >> 16).astype(np.uint16)   # truncate to bf16 bits
    else:
        lg = x
    masked = np.array([1, 1, 1, 0, 1, 1], np.uint8)
    full = oracle.stats(lg, masked)
    parts, offs = _shard_stats(lg, masked, sizes)
    m = oracle.merge_shard_stats(parts, offs)
    assert np.array_equal(m.argmax, full.argmax)
    assert np.array_equal(m.row_max, full.row_max)
    act = masked.astype(bool)
    assert np.allclose(m.lse[act], full.lse[act], rtol=1e-12, atol=0)
    assert np.allclose(m.conf[act], full.conf[act], rtol=1e-12, atol=0)
    assert np.all(np.isneginf(m.lse[~act])) and np.all(m.conf[~act] == 0)
    assert np.all(m.argmax[~act] == -1)


def test_shard_offsets_matter():
    # a merge that forgot the offsets would return the local index 0 here
    rng = np.random.default_rng(3)
    x = rng.normal(0, 1, size=(1, 40)).astype(np.float32)
    x[0, 30] = 7.0
    parts, offs = _shard_stats(x, None, [20, 20])
    m = oracle.merge_shard_stats(parts, offs)
    assert m.argmax[0] == 30
