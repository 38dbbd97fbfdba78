"""GPU parity of the gated MLP (st_gated_mlp) against the float64 oracle.

h = silu(x W1^T) * (x W3^T), y = h W2^T, with bf16 x and weights, and fp32 accumulation in both tensor-core GEMMs.
This is TSP's feed-forward layer (TSP summary, section 2, gated MLP layer).

The kernel holds h in bf16. Bounds on the two outputs:
- h: within half a bf16 ulp of the exact value, plus the fp32 accumulation error of the two dot products.
  Half an ulp is at most 2^-8 of the value's magnitude; the accumulation error is held to 1e-4 of h's RMS.
- y in fp32: compared with the oracle run on the same bf16 rounding of h.
  - The bounds are the bf16 ones: max error 1e-2 and mean error 1e-3 of y's RMS.
  - An element of h whose fp32 value lies within the fp32 accumulation error of a bf16 rounding boundary can round
    the other way. That moves y by one bf16 ulp of the element times its W2 weight: about 1e-3 of the RMS at F = 128.
    Over 4096-long dot products about 0.3 % of the elements of h do so, and the mean error of y reaches about 2e-4
    of its RMS.
- y in bf16: must be the fp32 y rounded once, bit for bit.
"""
import numpy as np
import pytest
import torch

import domain_ring_attention_gb300 as st
from oracle import mlp
from gpu_common import assert_no_device_error, f64

pytestmark = pytest.mark.gpu


def inputs(M, hidden, F, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((M, hidden), generator=g).to(torch.bfloat16)
    w1 = (torch.randn((F, hidden), generator=g) / hidden ** 0.5).to(torch.bfloat16)
    w3 = (torch.randn((F, hidden), generator=g) / hidden ** 0.5).to(torch.bfloat16)
    w2 = (torch.randn((hidden, F), generator=g) / F ** 0.5).to(torch.bfloat16)
    return x, w1, w3, w2


def check_h(h, h_ref):
    err = np.abs(f64(h) - h_ref)
    rms = float(np.sqrt(np.mean(h_ref * h_ref)))
    bound = 2.0 ** -8 * np.abs(h_ref) + 1e-4 * rms
    worst = int(np.argmax(err - bound))
    assert np.all(err <= bound), ("h", err.flat[worst], bound.flat[worst])


def check_y(y, y_ref):
    err = np.abs(f64(y) - y_ref)
    rms = float(np.sqrt(np.mean(y_ref * y_ref)))
    assert err.max() / rms <= 1e-2 and err.mean() / rms <= 1e-3, (err.max() / rms, err.mean() / rms)


def run(x, w1, w3, w2):
    xd, w1d, w3d, w2d = (t.cuda() for t in (x, w1, w3, w2))
    y32, h = st.st_gated_mlp(xd, w1d, w3d, w2d, out_dtype=torch.float32)
    y16, h2 = st.st_gated_mlp(xd, w1d, w3d, w2d, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert_no_device_error()
    assert torch.equal(h, h2)
    assert torch.equal(y16, y32.to(torch.bfloat16)), "bf16 output is not the fp32 output rounded once"
    return y32, h


# one tile; ragged M, hidden and F edges over several tiles; one row; a skinny F; a 7B-width layer slice
@pytest.mark.parametrize("M,hidden,F", [(128, 256, 128), (300, 264, 200), (1, 8, 8), (777, 520, 72),
                                        (1000, 1024, 2816), (512, 4096, 11008)])
def test_gated_mlp_matches_oracle(M, hidden, F):
    x, w1, w3, w2 = inputs(M, hidden, F, seed=M + hidden + F)
    y, h = run(x, w1, w3, w2)
    _, h_ref = mlp.gated_mlp(f64(x), f64(w1), f64(w3), f64(w2))
    check_h(h, h_ref)
    y_ref, _ = mlp.gated_mlp(f64(x), f64(w1), f64(w3), f64(w2), round_h=mlp.round_bf16)
    check_y(y, y_ref)


def test_gated_mlp_full_size_sampled():
    """The 7B-style layer (hidden 4096 = 32 heads x 128, F = 11008) over 65536 tokens, checked on sampled rows."""
    M, hidden, F = 65536, 4096, 11008
    x, w1, w3, w2 = inputs(M, hidden, F, seed=6)
    y, h = run(x, w1, w3, w2)
    rows = np.random.default_rng(1).choice(M, 96, replace=False)
    idx = torch.as_tensor(rows).cuda()
    _, h_ref = mlp.gated_mlp(f64(x[rows]), f64(w1), f64(w3), f64(w2))
    check_h(h[idx], h_ref)
    y_ref, _ = mlp.gated_mlp(f64(x[rows]), f64(w1), f64(w3), f64(w2), round_h=mlp.round_bf16)
    check_y(y[idx], y_ref)


def test_ring_partials_sum_to_the_layer():
    """The pages' ring schedule on the GPU: each weight shard's partial output (rows F_j of W1 and W3, columns F_j
    of W2), computed by its own call, summed over the shards, equals the one-call layer within fp32 rounding; h of
    each shard is the same columns of the full h, bit for bit."""
    M, hidden, F = 640, 512, 1216
    x, w1, w3, w2 = inputs(M, hidden, F, seed=12)
    xd, w1d, w3d, w2d = (t.cuda() for t in (x, w1, w3, w2))
    full, h_full = st.st_gated_mlp(xd, w1d, w3d, w2d, out_dtype=torch.float32)
    shards = [400, 8, 520, 288]
    fo = np.cumsum([0] + shards)
    acc = torch.zeros_like(full)
    for j in range(len(shards)):
        cols = slice(int(fo[j]), int(fo[j + 1]))
        part, h_j = st.st_gated_mlp(xd, w1d[cols].contiguous(), w3d[cols].contiguous(), w2d[:, cols].contiguous(),
                                    out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert torch.equal(h_j, h_full[:, cols])
        acc += part
    torch.cuda.synchronize()
    assert_no_device_error()
    rms = float(full.pow(2).mean().sqrt())
    assert float((acc - full).abs().max()) <= 1e-5 * rms
