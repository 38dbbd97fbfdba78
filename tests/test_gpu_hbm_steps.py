"""The backward's bandwidth-bound steps called on their own through the C-ABI: Delta (the row sums of dO o O),
the fp32 -> bf16 conversion of an accumulator, and the exact fp16 operand copy the tensor-core kernels run on."""
import numpy as np
import pytest
import torch

from domain_ring_attention_gb300 import _lib
from domain_ring_attention_gb300.workloads import Workload, make_inputs
from gpu_common import f64
from oracle import attention as oa

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("out_f32", [True, False])
def test_delta_matches_the_oracle(d, out_f32):
    lens = (300, 212, 512)
    wl = Workload("delta", B=2, H=3, d=d, lens=lens, causal=True, zigzag=True, dtype="bf16")
    q, k, v, do = make_inputs(wl, seed=8, with_dout=True)
    outs, _, deltas = oa.row_stats(f64(q), f64(k), f64(v), f64(do), lens, True, True)
    ref_out = np.stack([np.stack([outs[(b, h)] for h in range(3)], axis=1) for b in range(2)])   # [B,S,H,d]
    out_t = torch.from_numpy(ref_out).float()
    if not out_f32:
        out_t = out_t.to(torch.bfloat16)
    got = _lib.st_attn_bwd_delta(out_t.cuda(), do.cuda())
    torch.cuda.synchronize()
    # Delta of the values handed to the kernel, in float64
    ref = np.einsum("bshc,bshc->bhs", f64(out_t), f64(do))
    assert np.abs(f64(got) - ref).max() <= 1e-5 * max(1.0, np.abs(ref).max())
    if out_f32:   # and the oracle's own Delta of its float64 output, within fp32 rounding of out
        ref2 = np.stack([np.stack([deltas[(b, h)] for h in range(3)]) for b in range(2)])
        assert np.abs(f64(got) - ref2).max() <= 1e-4


def test_convert_rounds_to_nearest_even():
    g = torch.Generator().manual_seed(4)
    x = torch.randn(3 * 1024 + 8, generator=g) * 100
    x[:8] = torch.tensor([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -0.0, 0.0, 65504.0, 1e-40, -1e38, 3.0e38])   # ties, zeros, tiny, big
    got = _lib.st_convert_f32(x.cuda(), torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(got.cpu().view(torch.int16), x.to(torch.bfloat16).view(torch.int16))


@pytest.mark.parametrize("scale", [1.0, 1e-3, 3e4])
def test_fp16_scaled_copy_is_exact(scale):
    g = torch.Generator().manual_seed(6)
    x = (torch.randn(4096 * 8, generator=g) * scale).to(torch.bfloat16)
    y, e = _lib.st_fp16_scaled_copy(x.cuda())
    torch.cuda.synchronize()
    ev = int(e[0].item())
    amax = float(x.float().abs().max())
    assert 2.0 ** 13 <= amax * 2.0 ** -ev < 2.0 ** 14
    back = y.cpu().double() * 2.0 ** ev
    normal = x.double().abs() * 2.0 ** -ev >= 2.0 ** -14        # values in fp16's normal range after scaling
    assert torch.equal(back[normal], x.double()[normal])
