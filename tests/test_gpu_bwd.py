"""GPU parity of the backward path against the float64 oracle, through the C-ABI."""
import pytest
import torch

import domain_ring_attention_gb300 as st
from domain_ring_attention_gb300.workloads import WORKLOADS, Workload
from gpu_common import assert_close, check_full, f64, run_case
from oracle import attention as oa

pytestmark = pytest.mark.gpu

SMALL = [
    ((100, 150, 130, 132), False, False),
    ((100, 150, 130, 132), False, True),
    ((1, 7, 64, 129), False, True),
    ((300,), False, True),
    ((2, 6, 250, 32), True, True),
    ((128, 128, 128, 128), True, True),
    ((192, 64, 320, 128), True, False),
    ((512, 256, 768, 512), True, True),
]


def test_tiny_fp32_workload():
    wl = WORKLOADS["tiny_fp32"]
    check_full(wl, run_case(wl))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("lens,zigzag,causal", SMALL)
def test_small_layouts_backward(lens, zigzag, causal, d, dtype):
    wl = Workload("small", B=2, H=2, d=d, lens=lens, causal=causal, zigzag=zigzag, dtype=dtype)
    check_full(wl, run_case(wl, seed=sum(lens) + d))


def test_bf16_gradients_in_bf16():
    wl = Workload("small", B=1, H=3, d=128, lens=(256, 128, 384), causal=True, zigzag=True,
                  dtype="bf16")
    res32 = run_case(wl, seed=3)
    res16 = run_case(wl, seed=3, grad_dtype=torch.bfloat16)
    for g16, g32 in zip(res16["grads"], res32["grads"]):
        assert g16.dtype == torch.bfloat16
        # the bf16 gradients are the fp32 ones rounded once (within one bf16 ulp,
        # since fp32 accumulation order may differ between runs)
        torch.testing.assert_close(g16.float(), g32, rtol=2.0 ** -7, atol=1e-6 * g32.abs().max().item())


def test_backward_with_bf16_out():
    """The backward also accepts the forward output in bf16 (Delta then carries
    its rounding); on a non-causal case the gradients still meet the bound."""
    wl = Workload("bf16out", B=1, H=2, d=64, lens=(384, 640), causal=False, zigzag=False, dtype="bf16")
    res = run_case(wl, seed=21, backward=False)
    q, k, v, do = res["in"]
    lay = st.Layout(wl.lens)
    grads = st.st_attn_bwd(lay, q, k, v, res["out_native"], res["lse"], do)
    torch.cuda.synchronize()
    Q, K, V, DO = (f64(x) for x in (q, k, v, do))
    ro, rl = oa.forward(Q, K, V, wl.lens)
    rg = oa.backward(Q, K, V, ro, rl, DO, wl.lens)
    for name, g, r in zip(("dq", "dk", "dv"), grads, rg):
        assert_close(f64(g), r, "bf16", name, rel_rms=True)


def test_vit1024_workload_backward_full():
    wl = WORKLOADS["vit1024_s4096"]
    check_full(wl, run_case(wl), backward=True)


@pytest.mark.slow
def test_train_workload_backward_one_head():
    wl = WORKLOADS["train_s32768"]
    res = run_case(wl, backward=True)
    b, h = 1, 5
    q, k, v, do = (f64(x[b:b + 1, :, h:h + 1]) for x in res["in"])
    ro, rl = oa.forward(q, k, v, wl.lens, wl.zigzag, wl.causal)
    rg = oa.backward(q, k, v, ro, rl, do, wl.lens, wl.zigzag, wl.causal)
    for name, g, r in zip(("dq", "dk", "dv"), res["grads"], rg):
        assert_close(f64(g[b:b + 1, :, h:h + 1]), r, wl.dtype, name, rel_rms=True)
