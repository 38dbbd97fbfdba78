"""GPU parity of the halo exchange and the sharded 2-D convolution against the float64 oracle.

ShardTensor summary, section 2, communication: the halo exchange lets a convolution over a row-sharded image, with
uneven shards, give the numbers of the layer on the whole image.

Checks:
- The exchange is byte work. After it, every padded shard must equal the oracle's padded chunk bit for bit; the
  pad rows start out filled with a sentinel value.
- The convolution's fp32 output is held to max 1e-3 and mean 1e-4 of the oracle's RMS. fp32 accumulation over
  k*k*C_in products drifts by a few 1e-6 of the RMS.
- The bf16 output must be the fp32 output rounded once, bit for bit.
- The outputs stacked in shard order must match the oracle's convolution of the whole image.
"""
import numpy as np
import pytest
import torch

import domain_ring_attention_gb300 as st
from domain_ring_attention_gb300.workloads import dirichlet_shard_lengths
from oracle import halo
from gpu_common import assert_no_device_error, f64

pytestmark = pytest.mark.gpu

SENTINEL = 1000.0


def make(H, W, C_in, C_out, k, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((H, W, C_in), generator=g).to(torch.bfloat16)
    w = (torch.randn((C_out, k, k, C_in), generator=g) / (k * k * C_in) ** 0.5).to(torch.bfloat16)
    b = torch.randn((C_out,), generator=g) * 0.1
    return x, w, b


def padded_shards(x, rows, h):
    """Each shard's own rows in a [L + 2h, W, C] device buffer whose pad rows hold a sentinel."""
    off = np.cumsum([0] + list(rows))
    out = []
    for r, L in enumerate(rows):
        t = torch.full((L + 2 * h, x.shape[1], x.shape[2]), SENTINEL, dtype=torch.bfloat16, device="cuda")
        t[h:h + L] = x[off[r]:off[r + 1]].cuda()
        out.append(t)
    return out


def check(y, ref):
    err = np.abs(f64(y) - ref)
    rms = float(np.sqrt(np.mean(ref * ref)))
    assert err.max() / rms <= 1e-3 and err.mean() / rms <= 1e-4, (err.max() / rms, err.mean() / rms)


@pytest.mark.parametrize("rows,W,C_in,C_out,k", [
    ([5, 1, 7], 40, 64, 64, 3),            # a one-row shard, W below one pixel tile
    ([3, 1, 1, 1, 6], 130, 64, 136, 5),    # halo reaching two shards away, ragged W and C_out
    ([12], 128, 128, 256, 1),              # one shard, pointwise
    ([8, 9], 300, 192, 264, 7),            # two channel tiles (256 + 8), three pixel tiles
    ([2, 2], 1, 64, 8, 3),                 # one pixel wide, eight channels
])
def test_halo_and_conv_match_oracle(rows, W, C_in, C_out, k):
    h = (k - 1) // 2
    x, w, b = make(sum(rows), W, C_in, C_out, k, seed=sum(rows) * 7 + W + k)
    shards = padded_shards(x, rows, h)
    st.st_halo_exchange(shards, h)
    torch.cuda.synchronize()
    ref_pad = halo.halo_exchange(halo.split_rows(f64(x), rows), h)
    for got, ref in zip(shards, ref_pad):
        np.testing.assert_array_equal(f64(got), ref)
    wd, bd = w.cuda(), b.cuda()
    y32 = st.st_conv2d_sharded(shards, wd, bd, out_dtype=torch.float32)
    y16 = st.st_conv2d_sharded(shards, wd, bd, out_dtype=torch.bfloat16)
    y_nb = st.st_conv2d_sharded(shards, wd, None, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert_no_device_error()
    ref_local = [halo.conv_local(p, f64(w), f64(b)) for p in ref_pad]
    for a, a16, a_nb, ref in zip(y32, y16, y_nb, ref_local):
        check(a, ref)
        assert torch.equal(a16, a.to(torch.bfloat16)), "bf16 output is not the fp32 output rounded once"
        check(a_nb + bd, ref)
    check(torch.cat(y32), halo.conv2d(f64(x), f64(w), f64(b)))


def test_conus_grid_full_size_sampled():
    """The CONUS grid (1024 x 1792), 256 channels in and out, 3 x 3 kernel, four Dirichlet-uneven row shards.
    Checked on sampled rows: the first and last image rows, and the rows on both sides of every shard boundary,
    where the halo decides the result."""
    H, W, C, k = 1024, 1792, 256, 3
    rows = dirichlet_shard_lengths(H, 4, seed=0, multiple=1)
    g = torch.Generator(device="cuda").manual_seed(3)
    x = torch.randn((H, W, C), generator=g, device="cuda").to(torch.bfloat16)
    w = (torch.randn((C, k, k, C), generator=g, device="cuda") / (k * k * C) ** 0.5).to(torch.bfloat16)
    b = torch.randn((C,), generator=g, device="cuda") * 0.1
    shards = padded_shards(x, rows, 1)
    st.st_halo_exchange(shards, 1)
    y = torch.cat(st.st_conv2d_sharded(shards, w, b, out_dtype=torch.float32))
    torch.cuda.synchronize()
    assert_no_device_error()
    off = np.cumsum([0] + rows)
    sample = sorted({0, H - 1} | {int(o) + d for o in off[1:-1] for d in (-1, 0)})
    xp = torch.nn.functional.pad(x, (0, 0, 0, 0, 1, 1))      # one zero row above and below the image
    for i in sample:
        window = f64(xp[i:i + 3])                             # image rows i-1 .. i+1
        check(y[i:i + 1], halo.conv_local(window, f64(w), f64(b)))
