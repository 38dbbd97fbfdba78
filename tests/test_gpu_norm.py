"""GPU parity of the sharded group normalisation (st_group_norm_sharded) against the float64 oracle.

ShardTensor summary, section 2, communication: the statistics of every group are combined over all shards (the
all-reduce) before each shard normalises its own rows.

The oracle runs on the same bf16 input values.
- The fp32 output is held to max abs 1e-5, the bound for fp32 outputs. The statistics are exact to about 1e-7
  relative; the outputs are of order 1, at most about 6.
- The bf16 output must be the fp32 output rounded once, bit for bit.
- The rows outside the output's pad window must be left untouched.
"""
import numpy as np
import pytest
import torch

import domain_ring_attention_gb300 as st
from domain_ring_attention_gb300.workloads import dirichlet_shard_lengths
from oracle import norm
from gpu_common import assert_no_device_error, f64

pytestmark = pytest.mark.gpu


def make(rows, W, C, seed, loc=0.0):
    g = torch.Generator().manual_seed(seed)
    x = (loc + torch.randn((sum(rows), W, C), generator=g)).to(torch.bfloat16)
    gamma = 1.0 + 0.2 * torch.randn((C,), generator=g)
    beta = 0.1 * torch.randn((C,), generator=g)
    return x, gamma, beta


def shards_of(x, rows):
    off = np.cumsum([0] + list(rows))
    return [x[off[r]:off[r + 1]].contiguous().cuda() for r in range(len(rows))]


@pytest.mark.parametrize("rows,W,C,G,loc", [
    ([5, 1, 7], 40, 64, 8, 0.0),           # a one-row shard
    ([3, 1, 1, 1, 6], 130, 256, 32, 3.0),  # an offset mean (shifted sums), five shards
    ([12], 9, 8, 1, -2.0),                 # one shard, one group of 8 channels
    ([8, 9], 300, 2048, 16, 0.5),          # the widest C, 128 channels per group
    ([2, 2], 1, 128, 16, 0.0),             # one pixel wide
])
def test_group_norm_matches_oracle(rows, W, C, G, loc):
    x, gamma, beta = make(rows, W, C, seed=sum(rows) + W + C, loc=loc)
    xs = shards_of(x, rows)
    gd, bd = gamma.cuda(), beta.cuda()
    y32 = st.st_group_norm_sharded(xs, G, gd, bd, out_dtype=torch.float32)
    y16 = st.st_group_norm_sharded(xs, G, gd, bd, out_dtype=torch.bfloat16)
    y1 = st.st_group_norm_sharded(xs, G, None, None, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert_no_device_error()
    ref = norm.sharded_group_norm(f64(x), rows, G, f64(gamma), f64(beta))
    ref1 = norm.sharded_group_norm(f64(x), rows, G)
    for a, a16, b, r, r1 in zip(y32, y16, y1, ref, ref1):
        assert np.abs(f64(a) - r).max() <= 1e-5
        assert np.abs(f64(b) - r1).max() <= 1e-5
        assert torch.equal(a16, a.to(torch.bfloat16)), "bf16 output is not the fp32 output rounded once"
    np.testing.assert_allclose(np.concatenate([f64(a) for a in y32]),
                               norm.group_norm(f64(x), G, f64(gamma), f64(beta)), rtol=0, atol=1e-5)


def test_padded_output_feeds_the_convolution_layout():
    """out_pad rows are left alone, own rows land between them (the layout st_halo_exchange expects)."""
    rows, W, C, G = [4, 2, 5], 33, 64, 4
    x, gamma, beta = make(rows, W, C, seed=21)
    xs = shards_of(x, rows)
    gd, bd = gamma.cuda(), beta.cuda()
    o16 = [torch.full((L + 2, W, C), 7.0, device="cuda", dtype=torch.bfloat16) for L in rows]
    o32 = [torch.full((L + 2, W, C), 7.0, device="cuda", dtype=torch.float32) for L in rows]
    st.st_group_norm_sharded(xs, G, gd, bd, out=o16, out_pad=1)
    st.st_group_norm_sharded(xs, G, gd, bd, out=o32, out_pad=1)
    torch.cuda.synchronize()
    assert_no_device_error()
    ref = norm.sharded_group_norm(f64(x), rows, G, f64(gamma), f64(beta))
    for a16, a32, r in zip(o16, o32, ref):
        for a in (a16, a32):
            assert torch.all(a[0] == 7.0) and torch.all(a[-1] == 7.0)
        assert np.abs(f64(a32[1:-1]) - r).max() <= 1e-5
        assert torch.equal(a16[1:-1], a32[1:-1].to(torch.bfloat16))


def test_conus_grid_full_size():
    """The CONUS grid (1024 x 1792, 256 channels, 32 groups) over four Dirichlet-uneven row shards, checked on
    sampled rows (the first and last rows and both sides of every shard boundary) against the oracle's local
    statistics, all-reduce and normalisation of the whole input."""
    H, W, C, G = 1024, 1792, 256, 32
    rows = dirichlet_shard_lengths(H, 4, seed=0, multiple=1)
    g = torch.Generator(device="cuda").manual_seed(5)
    x = (1.0 + torch.randn((H, W, C), generator=g, device="cuda")).to(torch.bfloat16)
    gamma = 1.0 + 0.2 * torch.randn((C,), generator=g, device="cuda")
    beta = 0.1 * torch.randn((C,), generator=g, device="cuda")
    off = np.cumsum([0] + rows)
    xs = [x[off[r]:off[r + 1]] for r in range(len(rows))]
    y = torch.cat(st.st_group_norm_sharded(xs, G, gamma, beta, out_dtype=torch.float32))
    torch.cuda.synchronize()
    assert_no_device_error()
    xc = f64(x)
    stats = norm.all_reduce([norm.local_stats(xc[off[r]:off[r + 1]], G) for r in range(len(rows))])
    sample = sorted({0, H - 1} | {int(o) + d for o in off[1:-1] for d in (-1, 0)})
    ref = norm.normalize(xc[sample], stats, G, f64(gamma), f64(beta))
    assert np.abs(f64(y[torch.as_tensor(sample).cuda()]) - ref).max() <= 1e-5
