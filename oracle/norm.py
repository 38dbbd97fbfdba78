"""Oracle group normalisation over a spatially sharded image.

Test infrastructure only (see the package docstring).  float64 throughout.

ShardTensor summary, "ShardTensor" section 2, implementation details,
communication: normalisation over an input whose spatial axes are split over
devices needs collectives (an all-reduce) so that the sharded layer gives the
numbers of the layer on the whole input; the chunks may be uneven (sharding
shapes).

The pages name no normalisation. The reading here is group normalisation, the
normalisation of convolutional layers whose statistics span the spatial axes.
- The image is channels last, x [H, W, C], with C split into G groups of C/G channels.
- Group g has mean mu_g and biased variance var_g over every pixel and every channel of the group.
- The output is y[i, j, c] = (x[i, j, c] - mu_g) / sqrt(var_g + eps) * gamma[c] + beta[c].

Sharded over rows:
- every shard first computes its local statistics (count, mean and sum of squared deviations per group);
- an all-reduce then combines them by the pairwise rule for means and squared deviations (Chan, Golub and LeVeque);
- every shard normalises its own rows with the combined statistics.
Stacked in order, the shards' outputs equal the layer on the whole image.
"""
from __future__ import annotations

import numpy as np


def _groups(x, G):
    x = np.asarray(x, dtype=np.float64)
    H, W, C = x.shape
    if C % G:
        raise ValueError("C must be a multiple of G")
    return x.reshape(H * W, G, C // G)


def group_norm(x, G, gamma=None, beta=None, eps=1e-5):
    """The layer on the whole image, by its definition."""
    x = np.asarray(x, dtype=np.float64)
    xg = _groups(x, G)
    mu = xg.mean(axis=(0, 2))
    var = ((xg - mu[None, :, None]) ** 2).mean(axis=(0, 2))
    y = ((xg - mu[None, :, None]) / np.sqrt(var + eps)[None, :, None]).reshape(x.shape)
    C = x.shape[2]
    g = np.ones(C) if gamma is None else np.asarray(gamma, dtype=np.float64)
    b = np.zeros(C) if beta is None else np.asarray(beta, dtype=np.float64)
    return y * g + b


def local_stats(chunk, G):
    """One shard's statistics per group: (count, mean[G], M2[G]), M2 the sum
    of squared deviations from the shard's own mean."""
    xg = _groups(chunk, G)
    n = xg.shape[0] * xg.shape[2]
    mean = xg.mean(axis=(0, 2))
    m2 = ((xg - mean[None, :, None]) ** 2).sum(axis=(0, 2))
    return n, mean, m2


def combine(a, b):
    """Pairwise combination of two sets of statistics (Chan, Golub, LeVeque):
    n = n_a + n_b, delta = mean_b - mean_a, mean = mean_a + delta n_b / n,
    M2 = M2_a + M2_b + delta^2 n_a n_b / n."""
    na, ma, qa = a
    nb, mb, qb = b
    n = na + nb
    delta = mb - ma
    return n, ma + delta * (nb / n), qa + qb + delta * delta * (na * nb / n)


def all_reduce(stats):
    """Every shard's statistics combined, in shard order (what every rank
    holds after the all-reduce)."""
    out = stats[0]
    for s in stats[1:]:
        out = combine(out, s)
    return out


def sharded_group_norm(x, shard_rows, G, gamma=None, beta=None, eps=1e-5):
    """Local statistics, all-reduce, local normalisation: the list of the
    shards' outputs."""
    x = np.asarray(x, dtype=np.float64)
    off = np.concatenate([[0], np.cumsum(shard_rows)]).astype(int)
    if off[-1] != len(x) or min(shard_rows) < 1:
        raise ValueError("shard lengths must be >= 1 and cover the rows")
    chunks = [x[off[r]:off[r + 1]] for r in range(len(shard_rows))]
    stats = all_reduce([local_stats(c, G) for c in chunks])
    return [normalize(c, stats, G, gamma, beta, eps) for c in chunks]


def normalize(chunk, stats, G, gamma=None, beta=None, eps=1e-5):
    """Rows of one shard normalised with the combined statistics (n, mean, M2)."""
    n, mean, m2 = stats
    rstd = 1.0 / np.sqrt(m2 / n + eps)
    chunk = np.asarray(chunk, dtype=np.float64)
    C = chunk.shape[2]
    g = np.ones(C) if gamma is None else np.asarray(gamma, dtype=np.float64)
    b = np.zeros(C) if beta is None else np.asarray(beta, dtype=np.float64)
    y = ((_groups(chunk, G) - mean[None, :, None]) * rstd[None, :, None]).reshape(chunk.shape)
    return y * g + b
