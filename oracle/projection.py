"""Oracle projections: the linear layers on either side of the attention.

Test infrastructure only (see the package docstring).  float64 throughout;
numpy matmul is the only library step.

TSP summary, "Folding Tensor and Sequence Parallelism", section 2, attention
layer (broadcast schedule): every rank holds one shard of the sequence and one
shard of the packed weights W_Q, W_K, W_V, W_O; the ranks take turns, each
broadcasting its weight shard, and every rank computes the projections of its
own sequence shard with the weight shard of that turn.  ``broadcast_schedule``
follows those steps: for each weight shard in turn (the broadcast), for each
sequence shard (every rank), the local product of that block.  Taken over all
turns and ranks the blocks tile the whole output, which is the plain
definition ``project``:

    y[i, n] = sum_k x[i, k] w[n, k]      (x: [M, K] tokens, w: [N, K] a Linear
                                           layer's [out, in] weight)

For the input projections x holds the tokens ([B*S, hidden], buffer order) and
w the packed [3*H*d, hidden] W_Q|W_K|W_V, so y viewed as [B, S, 3, H, d] holds
q, k and v; for the output projection x is the attention output [B*S, H*d]
and w is W_O [hidden, H*d].
"""
from __future__ import annotations

import numpy as np


def project(x, w):
    """y = x w^T in float64 (the definition)."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    return x @ w.T


def broadcast_schedule(x, w, seq_lens, weight_lens):
    """The broadcast schedule on D ranks: seq_lens splits the rows of x (the
    sequence shards), weight_lens the rows of w (the weight shards, i.e. the
    output columns).  Turn t broadcasts weight shard t; every rank r computes
    its block x_r w_t^T.  Returns the assembled output and the list of
    (turn, rank) blocks in the order they are computed."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    so = np.concatenate([[0], np.cumsum(seq_lens)]).astype(int)
    wo = np.concatenate([[0], np.cumsum(weight_lens)]).astype(int)
    if so[-1] != x.shape[0] or wo[-1] != w.shape[0]:
        raise ValueError("shard lengths do not cover the tensors")
    y = np.zeros((x.shape[0], w.shape[0]))
    order = []
    for t in range(len(weight_lens)):                  # turn t: rank t broadcasts its weight shard
        w_t = w[wo[t]:wo[t + 1]]
        for r in range(len(seq_lens)):                 # every rank: its sequence shard x its copy of w_t
            y[so[r]:so[r + 1], wo[t]:wo[t + 1]] = x[so[r]:so[r + 1]] @ w_t.T
            order.append((t, r))
    return y, order


def split_qkv(y, B, S, H, d):
    """View the input projection's output [B*S, 3*H*d] as q, k, v [B, S, H, d]."""
    y = np.asarray(y).reshape(B, S, 3, H, d)
    return y[:, :, 0], y[:, :, 1], y[:, :, 2]
