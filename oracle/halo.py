"""Oracle halo exchange and 2-D convolution over a spatially sharded image.

Test infrastructure only (see the package docstring).  float64 throughout;
numpy's matmul is the only library step.

ShardTensor summary, "ShardTensor" section 2, implementation details,
communication: on an input whose spatial axes are split over devices, a
convolution or a normalisation needs the pixels next to each chunk that
neighbouring devices hold (the "halo") so that the sharded layer gives the same
numbers as the layer on the whole input.  The split may be uneven: the
sharding shapes give each chunk's own length (section 2, dynamic shapes).

The pages fix neither the convolution nor its layout.  This module reads it as
the convolution of deep-learning layers:
- a 2-D cross-correlation, stride 1, odd kernel size k, zero padding h = (k - 1) / 2 on every side (the output is
  as large as the input);
- channels last;
- x is [H, W, C_in], w is [C_out, k, k, C_in] and the bias is [C_out]:

    y[i, j, o] = bias[o] + sum_{u, v, c} x[i + u - h, j + v - h, c] w[o, u, v, c],
    where x is taken as 0 outside the image.

The H rows are split into D shards of lengths L_r, in order.
- ``halo_exchange`` gives every shard its padded local chunk: image rows off_r - h ... off_r + L_r + h - 1. Each
  row is taken from whichever shard owns it. A shard shorter than h draws its halo from shards further away.
  Rows outside the image are zero.
- ``conv_local`` convolves one padded chunk. It is valid along the rows (the halo supplies them) and zero-padded
  along W.
- The local outputs, stacked in shard order, equal ``conv2d`` of the whole image.
"""
from __future__ import annotations

import numpy as np


def _taps(xp, w, rows_out, W, bias):
    """Sum over the k*k taps of a row-padded, column-padded input."""
    C_out, k = w.shape[0], w.shape[1]
    y = np.zeros((rows_out, W, C_out))
    for u in range(k):
        for v in range(k):
            y += xp[u:u + rows_out, v:v + W, :] @ w[:, u, v, :].T
    if bias is not None:
        y += np.asarray(bias, dtype=np.float64)
    return y


def conv2d(x, w, bias=None):
    """The layer on the whole image, by its definition."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    k = w.shape[1]
    if k % 2 == 0 or w.shape[2] != k or w.shape[3] != x.shape[2]:
        raise ValueError("weight must be [C_out, k, k, C_in] with k odd")
    h = (k - 1) // 2
    H, W, _ = x.shape
    xp = np.pad(x, ((h, h), (h, h), (0, 0)))
    return _taps(xp, w, H, W, bias)


def split_rows(x, shard_rows):
    """The shards' own chunks (no halo): consecutive row ranges of lengths shard_rows."""
    off = np.concatenate([[0], np.cumsum(shard_rows)]).astype(int)
    if off[-1] != len(x) or min(shard_rows) < 1:
        raise ValueError("shard lengths must be >= 1 and cover the rows")
    return [np.asarray(x[off[r]:off[r + 1]], dtype=np.float64) for r in range(len(shard_rows))]


def halo_exchange(chunks, h):
    """Padded local chunks: chunk r with h rows above and h rows below, each
    taken from the shard that owns that image row (zero outside the image)."""
    lens = [len(c) for c in chunks]
    off = np.concatenate([[0], np.cumsum(lens)]).astype(int)
    H = int(off[-1])
    W, C = chunks[0].shape[1], chunks[0].shape[2]

    def image_row(g):
        if g < 0 or g >= H:
            return np.zeros((W, C))
        r = int(np.searchsorted(off, g, side="right")) - 1   # the shard that owns row g
        return chunks[r][g - off[r]]

    padded = []
    for r, c in enumerate(chunks):
        above = [image_row(off[r] - h + i) for i in range(h)]
        below = [image_row(off[r + 1] + i) for i in range(h)]
        padded.append(np.concatenate([np.reshape(above, (h, W, C)), c, np.reshape(below, (h, W, C))], axis=0))
    return padded


def conv_local(xp, w, bias=None):
    """One shard's output from its padded chunk [L + 2h, W, C_in]: [L, W, C_out]."""
    xp = np.asarray(xp, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    k = w.shape[1]
    h = (k - 1) // 2
    L = xp.shape[0] - 2 * h
    xpw = np.pad(xp, ((0, 0), (h, h), (0, 0)))
    return _taps(xpw, w, L, xp.shape[1], bias)


def sharded_conv2d(x, shard_rows, w, bias=None):
    """Split, exchange halos, convolve each shard: the list of local outputs."""
    h = (np.asarray(w).shape[1] - 1) // 2
    return [conv_local(p, w, bias) for p in halo_exchange(split_rows(x, shard_rows), h)]
