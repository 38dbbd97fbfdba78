"""GPU parity of the projection GEMM (st_proj_gemm) against the float64 oracle.

y = x w^T with bf16 x, w and fp32 accumulation (TSP summary, section 2,
attention layer: the QKV and output projections every rank computes for its
sequence shard with each packed weight shard).  The fp32 output is held to max
1e-3, mean 1e-4 of the oracle relative to the output's RMS (fp32 accumulation
of up to 4096 products of magnitude ~1/sqrt(K) drifts by a few 1e-6 of the
RMS per element), and the bf16 output must be that fp32 output rounded once
(bit for bit) -- an RMS-relative bound would not fit it: rounding an output
of 6x the RMS to bf16 alone moves it by up to 1.6e-2 of the RMS.
"""
import numpy as np
import pytest
import torch

import domain_ring_attention_gb300 as st
from oracle import projection
from gpu_common import assert_no_device_error, f64

pytestmark = pytest.mark.gpu


def inputs(M, N, K, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((M, K), generator=g).to(torch.bfloat16)
    w = (torch.randn((N, K), generator=g) / K ** 0.5).to(torch.bfloat16)
    return x, w


def check(y, ref, tol_max, tol_mean):
    err = np.abs(f64(y) - ref)
    rms = float(np.sqrt(np.mean(ref * ref)))
    assert err.max() / rms <= tol_max and err.mean() / rms <= tol_mean, (err.max() / rms, err.mean() / rms)


# one tile, several tiles with ragged M / N / K edges, one row, a skinny K
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (300, 264, 200), (1000, 3072, 1024), (1, 8, 8), (777, 520, 72),
                                   (2048, 768, 4096)])
def test_proj_matches_oracle(M, N, K):
    x, w = inputs(M, N, K, seed=M + N + K)
    ref = projection.project(f64(x), f64(w))
    xd, wd = x.cuda(), w.cuda()
    y32 = st.st_proj_gemm(xd, wd, out_dtype=torch.float32)
    y16 = st.st_proj_gemm(xd, wd, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert_no_device_error()
    check(y32, ref, 1e-3, 1e-4)
    assert torch.equal(y16, y32.to(torch.bfloat16)), "bf16 output is not the fp32 output rounded once"


def test_qkv_projection_full_size_sampled():
    """The ViT 4096^2 input projection (65536 tokens, hidden 1024 = 16 heads x
    64, packed W_Q|W_K|W_V [3072, 1024]) in buffer order, checked on sampled
    rows; its output split as [B, S, 3, H, d] gives q, k, v."""
    B, S, H, d = 1, 65536, 16, 64
    x, w = inputs(B * S, 3 * H * d, H * d, seed=5)
    xd, wd = x.cuda(), w.cuda()
    y = st.st_proj_gemm(xd.view(B, S, H * d), wd, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert_no_device_error()
    assert tuple(y.shape) == (B, S, 3 * H * d)
    rows = np.random.default_rng(0).choice(B * S, 256, replace=False)
    ref = projection.project(f64(x[rows]), f64(w))
    check(y.view(B * S, -1)[torch.as_tensor(rows).cuda()], ref, 1e-3, 1e-4)
    q, k, v = projection.split_qkv(f64(y[:, :8]), B, 8, H, d)
    yv = y.view(B, S, 3, H, d)
    np.testing.assert_array_equal(q, f64(yv[:, :8, 0]))
    np.testing.assert_array_equal(v, f64(yv[:, :8, 2]))


def test_shard_blocks_equal_the_full_product():
    """Each (sequence shard, weight shard) block of the broadcast schedule,
    computed on its own, equals the same block of the full product (the
    kernel's tiling is independent of how the pages' ranks would split the
    work)."""
    x, w = inputs(700, 528, 256, seed=9)
    xd, wd = x.cuda(), w.cuda()
    full = st.st_proj_gemm(xd, wd, out_dtype=torch.float32)
    seq, wts = [300, 100, 300], [264, 264]
    so, wo = np.cumsum([0] + seq), np.cumsum([0] + wts)
    for t in range(len(wts)):
        for r in range(len(seq)):
            blk = st.st_proj_gemm(xd[so[r]:so[r + 1]].contiguous(), wd[wo[t]:wo[t + 1]].contiguous(),
                                  out_dtype=torch.float32)
            torch.cuda.synchronize()
            torch.testing.assert_close(blk, full[so[r]:so[r + 1], wo[t]:wo[t + 1]], rtol=1e-6, atol=1e-6)
    assert_no_device_error()
