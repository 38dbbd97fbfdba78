"""Pins of the gated-MLP oracle (CPU only).

The oracle's layer is pinned by what does not re-type it:
- textbook values and identities of the logistic function;
- scipy's logistic routine;
- torch's bf16 conversion;
- a hand-worked example with printed constants (it fails if the gate is put on the W3 branch or W2 is transposed);
- pure-Python loops on tiny inputs;
- the invariant that the pages' ring schedule (TSP summary, section 2, gated MLP layer) assembles the same layer for
  any sharding of the tokens and of the hidden units, in either ring direction.
"""
import itertools
import math

import numpy as np
import pytest
import torch

from oracle import mlp


def test_silu_textbook_values():
    # sigmoid(1) = e / (1 + e) = 0.73105857863000487...
    assert mlp.silu(1.0) == pytest.approx(0.7310585786300049, rel=1e-15)
    assert mlp.silu(0.0) == 0.0
    # sigmoid(-1) = 1 - sigmoid(1)
    assert mlp.silu(-1.0) == pytest.approx(-(1 - 0.7310585786300049), rel=1e-14)


def test_silu_identities():
    a = np.linspace(-30, 30, 601)
    # sigmoid(a) + sigmoid(-a) = 1  =>  silu(a) - silu(-a) = a; a flipped exponent gives -a
    np.testing.assert_allclose(mlp.silu(a) - mlp.silu(-a), a, rtol=1e-12, atol=1e-12)
    # slope 1/2 at 0
    eps = 1e-6
    assert (mlp.silu(eps) - mlp.silu(-eps)) / (2 * eps) == pytest.approx(0.5, rel=1e-9)
    # limits: the identity for large a, zero (no NaN) for very negative a
    assert mlp.silu(800.0) == 800.0
    assert mlp.silu(-800.0) == 0.0 and not np.isnan(mlp.silu(-800.0))


def test_silu_matches_scipy_logistic():
    special = pytest.importorskip("scipy.special")
    a = np.random.default_rng(0).standard_normal(1000) * 8
    np.testing.assert_allclose(mlp.silu(a), a * special.expit(a), rtol=1e-13, atol=1e-300)


def test_round_bf16_matches_torch():
    rng = np.random.default_rng(1)
    a = np.concatenate([rng.standard_normal(5000) * 10.0 ** rng.integers(-6, 6, 5000),
                        # exact ties: 1 + 2^-8 rounds down to 1 (even), 1 + 3*2^-8 up to 1 + 2^-6
                        [1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 0.0, -0.0]])
    ref = torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(mlp.round_bf16(a), ref)
    assert mlp.round_bf16(1 + 2.0 ** -8) == 1.0
    assert mlp.round_bf16(1 + 3 * 2.0 ** -8) == 1 + 2.0 ** -6


def test_hand_worked_example():
    # x = [1, 2]; W1 = I -> a = [1, 2]; W3 = diag(3, -1) -> b = [3, -2]
    # h = [3 silu(1), -2 silu(2)] = [2.193175735890015, -3.5231883119115293]
    # W2 = [[1, 1], [2, 0]] -> y = [h0 + h1, 2 h0]
    x = np.array([[1.0, 2.0]])
    w1 = np.eye(2)
    w3 = np.diag([3.0, -1.0])
    w2 = np.array([[1.0, 1.0], [2.0, 0.0]])
    y, h = mlp.gated_mlp(x, w1, w3, w2)
    np.testing.assert_allclose(h, [[2.193175735890015, -3.5231883119115293]], rtol=1e-14)
    np.testing.assert_allclose(y, [[-1.3300125760215145, 4.38635147178003]], rtol=1e-14)


def loops(x, w1, w3, w2):
    M, hid, F = len(x), len(x[0]), len(w1)
    h = [[0.0] * F for _ in range(M)]
    for i in range(M):
        for f in range(F):
            a = sum(x[i][k] * w1[f][k] for k in range(hid))
            b = sum(x[i][k] * w3[f][k] for k in range(hid))
            h[i][f] = a / (1 + math.exp(-a)) * b
    return [[sum(h[i][f] * w2[n][f] for f in range(F)) for n in range(len(w2))] for i in range(M)]


def test_matches_python_loops():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((4, 6))
    w1, w3 = rng.standard_normal((2, 5, 6))
    w2 = rng.standard_normal((6, 5))
    y, _ = mlp.gated_mlp(x, w1, w3, w2)
    ref = loops(x.tolist(), w1.tolist(), w3.tolist(), w2.tolist())
    np.testing.assert_allclose(y, np.array(ref), rtol=1e-12, atol=1e-12)


def test_linear_in_up_and_down_weights_not_in_gate():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((7, 8))
    w1, w3, v3 = rng.standard_normal((3, 12, 8))
    w2, v2 = rng.standard_normal((2, 8, 12))
    y = lambda a, b, c: mlp.gated_mlp(x, a, b, c)[0]
    np.testing.assert_allclose(y(w1, 2 * w3 - v3, w2), 2 * y(w1, w3, w2) - y(w1, v3, w2), rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(y(w1, w3, w2 + v2), y(w1, w3, w2) + y(w1, w3, v2), rtol=1e-10, atol=1e-10)
    assert not np.allclose(y(2 * w1, w3, w2), 2 * y(w1, w3, w2))
    np.testing.assert_array_equal(mlp.gated_mlp(np.zeros((3, 8)), w1, w3, w2)[0], 0.0)


@pytest.mark.parametrize("direction", [1, -1])
@pytest.mark.parametrize("seq_lens,weight_lens", [
    ([5], [12]),
    ([3, 9], [4, 8]),
    ([7, 1, 4, 4], [1, 5, 3, 3]),
    ([2, 6, 1, 5, 3], [8, 1, 1, 1, 1]),
])
def test_ring_schedule_assembles_the_layer(seq_lens, weight_lens, direction):
    rng = np.random.default_rng(sum(seq_lens) * 31 + sum(weight_lens))
    M, F, hid = sum(seq_lens), sum(weight_lens), 6
    x = rng.standard_normal((M, hid))
    w1, w3 = rng.standard_normal((2, F, hid))
    w2 = rng.standard_normal((hid, F))
    y_ring, order = mlp.ring_schedule(x, w1, w3, w2, seq_lens, weight_lens, direction)
    y, _ = mlp.gated_mlp(x, w1, w3, w2)
    np.testing.assert_allclose(y_ring, y, rtol=1e-12, atol=1e-12)
    D = len(seq_lens)
    # every rank meets every weight shard once; step 0 uses its own shard
    assert sorted((r, j) for _, r, j in order) == sorted(itertools.product(range(D), range(D)))
    held = {(t, r): j for t, r, j in order}
    assert all(held[(0, r)] == r for r in range(D))
    # the shard a rank holds at step t is its neighbour's at step t + 1 (passed round the ring)
    for t in range(D - 1):
        for r in range(D):
            assert held[(t + 1, (r + direction) % D)] == held[(t, r)]


def test_ring_schedule_with_bf16_h_matches_definition():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((10, 16))
    w1, w3 = rng.standard_normal((2, 24, 16))
    w2 = rng.standard_normal((16, 24))
    y_ring, _ = mlp.ring_schedule(x, w1, w3, w2, [4, 6], [16, 8], round_h=mlp.round_bf16)
    y, h = mlp.gated_mlp(x, w1, w3, w2, round_h=mlp.round_bf16)
    np.testing.assert_allclose(y_ring, y, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(h, mlp.round_bf16(h))


def test_ring_schedule_rejects_bad_lengths():
    x = np.zeros((4, 2))
    w = np.zeros((6, 2))
    with pytest.raises(ValueError):
        mlp.ring_schedule(x, w, w, np.zeros((2, 6)), [2, 2], [3, 2])
    with pytest.raises(ValueError):
        mlp.ring_schedule(x, w, w, np.zeros((2, 6)), [2, 2], [6])
