"""Oracle gated MLP: the feed-forward layer that TSP runs with its ring schedule.

Test infrastructure only (see the package docstring).  float64 throughout;
numpy's matmul and exp are the only library steps.

TSP summary, "Folding Tensor and Sequence Parallelism", section 2, gated MLP
layer: the weight shards of W1, W2 and W3 travel round the ring of ranks
point to point; every rank keeps its own sequence shard and adds up the
partial outputs it computes with each shard as it passes, so the layer needs
no all-reduce.

The pages name the three weights but not the function.  The reading taken
here is the usual gated MLP with a SiLU gate on the W1 branch:

    a = x W1^T,  b = x W3^T                  x: [M, hidden]; W1, W3: [F, hidden]
    h = silu(a) * b,  silu(a) = a / (1 + e^-a)
    y = h W2^T                               W2: [hidden, F]

A weight shard j is a range F_j of the F hidden units: rows F_j of W1 and
W3, columns F_j of W2.  The columns F_j of h depend on shard j alone, so
y = sum_j (silu(x W1_j^T) * (x W3_j^T)) W2_j^T: the ring's partial outputs
add up to the whole layer, which is what ``ring_schedule`` checks.

``round_h`` (optional) is applied to h before the down projection: a path that
holds h in bf16 rounds it once there, and the oracle can model the same.
"""
from __future__ import annotations

import numpy as np


def silu(a):
    """a * sigmoid(a) = a / (1 + e^-a), float64.  For very negative a the
    exponential overflows to inf and the quotient is -0, its limit."""
    a = np.asarray(a, dtype=np.float64)
    with np.errstate(over="ignore"):
        return a / (1.0 + np.exp(-a))


def round_bf16(a):
    """Round float64 values to the nearest bf16 (ties to even), returned as
    float64.  The value is first rounded to float32 (ties to even), then the
    low 16 bits of the float32 pattern are rounded off; finite inputs only."""
    f = np.asarray(a, dtype=np.float64).astype(np.float32)
    bits = f.view(np.uint32).astype(np.uint64)
    keep = (bits + 0x7FFF + ((bits >> 16) & 1)) & 0xFFFF0000
    return keep.astype(np.uint32).view(np.float32).astype(np.float64)


def gated_mlp(x, w1, w3, w2, round_h=None):
    """The layer by its definition.  Returns (y [M, hidden], h [M, F])."""
    x = np.asarray(x, dtype=np.float64)
    w1 = np.asarray(w1, dtype=np.float64)
    w3 = np.asarray(w3, dtype=np.float64)
    w2 = np.asarray(w2, dtype=np.float64)
    h = silu(x @ w1.T) * (x @ w3.T)
    if round_h is not None:
        h = round_h(h)
    return h @ w2.T, h


def ring_schedule(x, w1, w3, w2, seq_lens, weight_lens, direction=1, round_h=None):
    """The ring schedule on D ranks.  seq_lens splits the rows of x (rank r
    keeps sequence shard r); weight_lens splits the F hidden units (rank r
    starts with weight shard r).  At step t every rank passes the shard it
    holds to its neighbour, so rank r holds shard (r - direction * t) mod D,
    computes that shard's partial output for its own tokens and adds it to
    its accumulator.  Returns the assembled y and the (step, rank, shard)
    triples in the order they are computed."""
    x = np.asarray(x, dtype=np.float64)
    w1 = np.asarray(w1, dtype=np.float64)
    w3 = np.asarray(w3, dtype=np.float64)
    w2 = np.asarray(w2, dtype=np.float64)
    D = len(seq_lens)
    if len(weight_lens) != D:
        raise ValueError("one weight shard per rank")
    so = np.concatenate([[0], np.cumsum(seq_lens)]).astype(int)
    fo = np.concatenate([[0], np.cumsum(weight_lens)]).astype(int)
    if so[-1] != x.shape[0] or fo[-1] != w1.shape[0]:
        raise ValueError("shard lengths do not cover the tensors")
    acc = [np.zeros((so[r + 1] - so[r], w2.shape[0])) for r in range(D)]
    order = []
    for t in range(D):
        for r in range(D):
            j = (r - direction * t) % D
            xr = x[so[r]:so[r + 1]]
            cols = slice(fo[j], fo[j + 1])
            h = silu(xr @ w1[cols].T) * (xr @ w3[cols].T)
            if round_h is not None:
                h = round_h(h)
            acc[r] += h @ w2[:, cols].T
            order.append((t, r, j))
    return np.concatenate(acc, axis=0), order
