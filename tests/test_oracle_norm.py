"""Pins of the sharded group-normalisation oracle (CPU only).

The definition is pinned against torch's float64 group_norm (NCHW) and by closed forms. With gamma = 1 and
beta = 0, every group of the output has mean 0 and variance var / (var + eps). A constant group gives beta.

The pairwise combination of statistics is pinned by the statistics of the concatenated data, and by invariance
under the order of combination.

The sharded layer is pinned by the pages' requirement (ShardTensor summary, section 2, communication): local
statistics, all-reduce, local normalisation equal the layer on the whole image, for uneven shards down to one row.
"""
import itertools

import numpy as np
import pytest
import torch

from oracle import norm


def rand(shape, seed, loc=0.0, scale=1.0):
    return loc + scale * np.random.default_rng(seed).standard_normal(shape)


@pytest.mark.parametrize("G", [1, 4, 16])
def test_group_norm_matches_torch(G):
    x = rand((6, 7, 16), G, loc=3.0, scale=2.0)
    gamma, beta = rand(16, 1), rand(16, 2)
    ref = torch.nn.functional.group_norm(torch.from_numpy(x).permute(2, 0, 1)[None], G,
                                         torch.from_numpy(gamma), torch.from_numpy(beta), eps=1e-5)
    np.testing.assert_allclose(norm.group_norm(x, G, gamma, beta), ref[0].permute(1, 2, 0).numpy(),
                               rtol=1e-12, atol=1e-12)


def test_closed_forms():
    x = rand((5, 4, 8), 3, loc=-7.0, scale=0.5)
    y = norm.group_norm(x, 2, eps=1e-5).reshape(-1, 2, 4)
    var = x.reshape(-1, 2, 4).var(axis=(0, 2))
    np.testing.assert_allclose(y.mean(axis=(0, 2)), 0.0, atol=1e-12)
    np.testing.assert_allclose(y.var(axis=(0, 2)), var / (var + 1e-5), rtol=1e-12)
    const = np.full((3, 3, 4), 2.5)
    beta = np.array([1.0, -2.0, 0.5, 4.0])
    np.testing.assert_allclose(norm.group_norm(const, 2, np.ones(4), beta), np.broadcast_to(beta, (3, 3, 4)))


def test_combine_matches_concatenation_in_any_order():
    parts = [rand((r, 3, 4), 10 + r, loc=r, scale=1 + r) for r in (1, 4, 2, 7)]
    whole = norm.local_stats(np.concatenate(parts), 2)
    stats = [norm.local_stats(p, 2) for p in parts]
    for perm in itertools.permutations(range(4)):
        n, mean, m2 = norm.all_reduce([stats[i] for i in perm])
        assert n == whole[0]
        np.testing.assert_allclose(mean, whole[1], rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(m2, whole[2], rtol=1e-12)


@pytest.mark.parametrize("shard_rows", [[9], [4, 5], [1, 3, 1, 4], [2, 1, 1, 1, 4]])
@pytest.mark.parametrize("G", [1, 8])
def test_sharded_equals_whole_image(shard_rows, G):
    H = sum(shard_rows)
    x = rand((H, 6, 16), H * 3 + G, loc=1.5)
    gamma, beta = rand(16, 4), rand(16, 5)
    local = norm.sharded_group_norm(x, shard_rows, G, gamma, beta)
    assert [len(y) for y in local] == shard_rows
    np.testing.assert_allclose(np.concatenate(local), norm.group_norm(x, G, gamma, beta), rtol=1e-12, atol=1e-12)


def test_local_statistics_alone_are_not_enough():
    # normalising each shard with its own statistics (no all-reduce) differs from the layer
    x = np.concatenate([rand((3, 4, 4), 6, loc=0.0), rand((3, 4, 4), 7, loc=5.0)])
    whole = norm.group_norm(x, 1)
    local_only = np.concatenate([norm.group_norm(x[:3], 1), norm.group_norm(x[3:], 1)])
    assert not np.allclose(whole, local_only)


def test_bad_shapes_are_refused():
    with pytest.raises(ValueError):
        norm.group_norm(np.zeros((2, 2, 6)), 4)
    with pytest.raises(ValueError):
        norm.sharded_group_norm(np.zeros((4, 2, 4)), [2, 1], 2)
