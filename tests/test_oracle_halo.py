"""Pins of the halo-exchange / sharded-convolution oracle (CPU only).

The definition is pinned against torch's float64 conv2d. A second pin is scipy's 2-D cross-correlation, summed
over channel pairs.
Further pins:
- pure-Python loops on a tiny input;
- a shifted-delta kernel, which fixes the orientation: cross-correlation, not a flipped convolution;
- the identity kernel and a box filter.

The sharded path is pinned by the pages' requirement (ShardTensor summary, section 2, communication): with the
halo exchanged, the sharded layer equals the layer on the whole image. This holds for uneven shards, including
shards shorter than the halo, and for every kernel size.
"""
import itertools

import numpy as np
import pytest
import torch

from oracle import halo


def rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


@pytest.mark.parametrize("k", [1, 3, 5])
def test_conv2d_matches_torch(k):
    x = rand((9, 11, 4), 0)
    w = rand((5, k, k, 4), 1)
    b = rand(5, 2)
    xt = torch.from_numpy(x).permute(2, 0, 1)[None]           # [1, C_in, H, W]
    wt = torch.from_numpy(w).permute(0, 3, 1, 2)              # [C_out, C_in, k, k]
    ref = torch.nn.functional.conv2d(xt, wt, torch.from_numpy(b), padding=(k - 1) // 2)[0].permute(1, 2, 0)
    np.testing.assert_allclose(halo.conv2d(x, w, b), ref.numpy(), rtol=1e-12, atol=1e-12)


def test_conv2d_matches_scipy_correlate():
    signal = pytest.importorskip("scipy.signal")
    x = rand((7, 8, 3), 3)
    w = rand((2, 3, 3, 3), 4)
    ref = np.zeros((7, 8, 2))
    for o, c in itertools.product(range(2), range(3)):
        ref[:, :, o] += signal.correlate2d(x[:, :, c], w[o, :, :, c], mode="same", boundary="fill")
    np.testing.assert_allclose(halo.conv2d(x, w), ref, rtol=1e-12, atol=1e-12)


def test_conv2d_matches_python_loops():
    x = rand((4, 5, 2), 5)
    w = rand((3, 3, 3, 2), 6)
    H, W, C = x.shape
    ref = np.zeros((H, W, 3))
    for i, j, o in itertools.product(range(H), range(W), range(3)):
        s = 0.0
        for u, v, c in itertools.product(range(3), range(3), range(C)):
            ii, jj = i + u - 1, j + v - 1
            if 0 <= ii < H and 0 <= jj < W:
                s += x[ii, jj, c] * w[o, u, v, c]
        ref[i, j, o] = s
    np.testing.assert_allclose(halo.conv2d(x, w), ref, rtol=1e-13, atol=1e-13)


def test_shifted_delta_kernel_fixes_orientation():
    # w[0, 0, 0, 0] = 1: y[i, j] = x[i - 1, j - 1] (a cross-correlation; a flipped kernel would give x[i + 1, j + 1])
    x = rand((6, 7, 1), 7)
    w = np.zeros((1, 3, 3, 1))
    w[0, 0, 0, 0] = 1.0
    y = halo.conv2d(x, w)
    np.testing.assert_array_equal(y[1:, 1:, 0], x[:-1, :-1, 0])
    np.testing.assert_array_equal(y[0, :, 0], 0.0)
    np.testing.assert_array_equal(y[:, 0, 0], 0.0)


def test_identity_and_box_kernels():
    x = rand((5, 6, 3), 8)
    ident = np.zeros((3, 3, 3, 3))
    for c in range(3):
        ident[c, 1, 1, c] = 1.0
    np.testing.assert_array_equal(halo.conv2d(x, ident), x)
    ones = np.ones((4, 5, 1))
    box = halo.conv2d(ones, np.ones((1, 3, 3, 1)))[:, :, 0]
    # interior pixels see 9 ones, edges 6, corners 4
    assert box[1, 1] == 9 and box[0, 2] == 6 and box[0, 0] == 4 and box[3, 4] == 4


@pytest.mark.parametrize("k", [1, 3, 5, 7])
@pytest.mark.parametrize("shard_rows", [[12], [5, 7], [1, 6, 2, 3], [3, 1, 1, 1, 6], [2, 2, 1, 7]])
def test_sharded_with_halo_equals_whole_image(shard_rows, k):
    H = sum(shard_rows)
    x = rand((H, 9, 3), H + k)
    w = rand((4, k, k, 3), k)
    b = rand(4, 11)
    local = halo.sharded_conv2d(x, shard_rows, w, b)
    assert [len(y) for y in local] == shard_rows
    np.testing.assert_allclose(np.concatenate(local), halo.conv2d(x, w, b), rtol=1e-12, atol=1e-12)


def test_halo_rows_come_from_the_owning_shards():
    x = np.arange(10, dtype=np.float64).reshape(10, 1, 1)      # row g holds the value g
    chunks = halo.split_rows(x, [1, 4, 1, 4])
    padded = halo.halo_exchange(chunks, 2)
    # shard 2 (row 5) reaches two rows into shards 1 and 3; shard 0 (row 0) sees zeros above
    np.testing.assert_array_equal(padded[2][:, 0, 0], [3, 4, 5, 6, 7])
    np.testing.assert_array_equal(padded[0][:, 0, 0], [0, 0, 0, 1, 2])
    np.testing.assert_array_equal(padded[3][:, 0, 0], [4, 5, 6, 7, 8, 9, 0, 0])


def test_without_halo_the_shard_edges_differ():
    # zero padding at every shard edge instead of the exchange changes the rows next to the cuts
    x = rand((8, 5, 2), 9)
    w = rand((2, 3, 3, 2), 10)
    chunks = halo.split_rows(x, [3, 5])
    no_halo = [halo.conv_local(np.pad(c, ((1, 1), (0, 0), (0, 0))), w) for c in chunks]
    whole = halo.conv2d(x, w)
    assert not np.allclose(no_halo[0][-1], whole[2])
    np.testing.assert_allclose(no_halo[0][:-1], whole[:2], rtol=1e-12, atol=1e-12)


def test_bad_shapes_are_refused():
    with pytest.raises(ValueError):
        halo.conv2d(np.zeros((3, 3, 2)), np.zeros((1, 2, 2, 2)))
    with pytest.raises(ValueError):
        halo.split_rows(np.zeros((4, 1, 1)), [2, 1])
    with pytest.raises(ValueError):
        halo.split_rows(np.zeros((4, 1, 1)), [4, 0])
