"""Brute-force attention with pure-Python loops, for tiny inputs only.

Test infrastructure only (see the package docstring).  Written from the
definition softmax(scale * Q K^T) V with no blocking, no shards and no numpy
arithmetic, for sequences of at most a few dozen rows.  Inputs are nested
lists (or arrays) in natural order, shape [S][d] for one (batch, head).
"""
from __future__ import annotations

import math


def attention(q, k, v, causal=False, scale=None):
    """Returns (out [S][d], lse [S]) for one head, natural order."""
    S = len(q)
    d = len(q[0])
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = []
    lse = []
    for i in range(S):
        scores = []
        for j in range(S):
            if causal and j > i:
                continue
            dot = 0.0
            for c in range(d):
                dot += float(q[i][c]) * float(k[j][c])
            scores.append((j, scale * dot))
        top = max(s for _, s in scores)
        tot = 0.0
        for _, s in scores:
            tot += math.exp(s - top)
        row_lse = top + math.log(tot)
        row = [0.0] * len(v[0])
        for j, s in scores:
            w = math.exp(s - row_lse)
            for c in range(len(v[0])):
                row[c] += w * float(v[j][c])
        out.append(row)
        lse.append(row_lse)
    return out, lse
