"""Oracle shard layout: sharding shapes and the zigzag re-partition.

Test infrastructure only (see the package docstring).

Sharding shapes (ShardTensor summary, section 2): every rank r of the sharded
axis holds a local chunk of its own length L_r; the chunks may be uneven.  The
sequence buffer holds shard 0's rows, then shard 1's, and so on, so shard r
occupies buffer rows [off[r], off[r+1]) with off the exclusive prefix sum.

Zigzag (TSP summary, section 2, attention layer): the sequence is cut into 2D
chunks in natural order and rank r holds chunks r and 2D-1-r, so that every
rank owns one early and one late piece and causal work is balanced.  The pages
only show the equal-length case; with uneven sharding shapes this oracle takes
chunk r and chunk 2D-1-r each of length L_r / 2 (L_r must be even), which is
the equal-length rule whenever all L_r are equal.  Rank r's buffer slab is
[chunk r ; chunk 2D-1-r] in that order.
"""
from __future__ import annotations

import numpy as np


def shard_offsets(lens) -> np.ndarray:
    """Exclusive prefix sum of the sharding shapes: off[0] = 0, off[D] = S."""
    lens = [int(x) for x in lens]
    if len(lens) < 1 or any(x < 1 for x in lens):
        raise ValueError("every shard needs at least one row")
    off = np.zeros(len(lens) + 1, dtype=np.int64)
    for r, L in enumerate(lens):
        off[r + 1] = off[r] + L
    return off


def zigzag_chunk_lengths(lens) -> np.ndarray:
    """Lengths of the 2D natural-order chunks: c_r = c_{2D-1-r} = L_r / 2."""
    D = len(lens)
    c = np.zeros(2 * D, dtype=np.int64)
    for r, L in enumerate(lens):
        if L % 2:
            raise ValueError("zigzag needs even shard lengths")
        c[r] = L // 2
        c[2 * D - 1 - r] = L // 2
    return c


def natural_positions(lens, zigzag: bool) -> np.ndarray:
    """pos[t] = natural (sequence) position of buffer row t."""
    off = shard_offsets(lens)
    S = int(off[-1])
    if not zigzag:
        return np.arange(S, dtype=np.int64)
    D = len(lens)
    c = zigzag_chunk_lengths(lens)
    chunk_start = np.concatenate([[0], np.cumsum(c)])
    pos = np.empty(S, dtype=np.int64)
    for r in range(D):
        half = int(lens[r]) // 2
        lo = int(off[r])
        pos[lo:lo + half] = chunk_start[r] + np.arange(half)
        pos[lo + half:lo + 2 * half] = chunk_start[2 * D - 1 - r] + np.arange(half)
    return pos


def shard_of_row(lens) -> np.ndarray:
    """owner[t] = the shard (rank) whose slab holds buffer row t."""
    off = shard_offsets(lens)
    owner = np.empty(int(off[-1]), dtype=np.int64)
    for r in range(len(lens)):
        owner[off[r]:off[r + 1]] = r
    return owner
