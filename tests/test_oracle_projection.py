"""Pins of the projection oracle (CPU only).

The oracle's `project` is a library matmul, so it is pinned against what does
not re-type it: a pure-Python triple loop on tiny inputs, the identity weight,
linearity, and the pages' broadcast schedule (TSP summary, section 2,
attention layer), which must assemble the same product for any sharding of
the sequence and of the weights.
"""
import itertools

import numpy as np
import pytest

from oracle import projection


def loops(x, w):
    M, K = len(x), len(x[0])
    N = len(w)
    return [[sum(float(x[i][k]) * float(w[n][k]) for k in range(K)) for n in range(N)] for i in range(M)]


def test_project_equals_triple_loop():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 7))
    w = rng.standard_normal((3, 7))
    np.testing.assert_allclose(projection.project(x, w), np.array(loops(x.tolist(), w.tolist())), rtol=1e-13,
                               atol=1e-13)


def test_identity_weight_returns_input():
    x = np.random.default_rng(1).standard_normal((9, 6))
    np.testing.assert_array_equal(projection.project(x, np.eye(6)), x)


def test_linear_in_x():
    rng = np.random.default_rng(2)
    x1, x2 = rng.standard_normal((2, 8, 5))
    w = rng.standard_normal((4, 5))
    lhs = projection.project(2.5 * x1 - 0.75 * x2, w)
    rhs = 2.5 * projection.project(x1, w) - 0.75 * projection.project(x2, w)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seq_lens,weight_lens", [([3, 1, 4, 2], [2, 5, 1, 4]), ([10], [12]), ([1, 1, 8], [6, 6, 1])])
def test_broadcast_schedule_assembles_the_product(seq_lens, weight_lens):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((sum(seq_lens), 6))
    w = rng.standard_normal((sum(weight_lens), 6))
    y, order = projection.broadcast_schedule(x, w, seq_lens, weight_lens)
    np.testing.assert_allclose(y, projection.project(x, w), rtol=1e-13, atol=1e-13)
    # one block per (turn, rank), turn-major: one broadcast per weight shard
    assert order == list(itertools.product(range(len(weight_lens)), range(len(seq_lens))))


def test_broadcast_schedule_rejects_bad_lengths():
    with pytest.raises(ValueError):
        projection.broadcast_schedule(np.zeros((4, 2)), np.zeros((3, 2)), [2, 1], [3])


def test_split_qkv_layout():
    """Output column n of the packed projection is (which, head, dim) = n
    split as [3, H, d]: with one-hot tokens the output rows are the weight's
    columns, so q/k/v come out as the three row blocks of w."""
    B, S, H, d = 1, 4, 2, 3
    hidden = B * S
    w = np.arange(3 * H * d * hidden, dtype=np.float64).reshape(3 * H * d, hidden)
    y = projection.project(np.eye(hidden), w)
    q, k, v = projection.split_qkv(y, B, S, H, d)
    for which, t in enumerate((q, k, v)):
        for s in range(S):
            np.testing.assert_array_equal(t[0, s].reshape(-1), w[which * H * d:(which + 1) * H * d, s])
