"""GPU parity of the forward path (fused ring forward, partials, merge,
permute) against the float64 oracle, through the C-ABI."""
import numpy as np
import pytest
import torch

import domain_ring_attention_gb300 as st
from domain_ring_attention_gb300.workloads import WORKLOADS, Workload, make_inputs, sample_rows
from gpu_common import assert_close, assert_lse, assert_no_device_error, check_full, check_rows, f64, run_case
from oracle import attention as oa
from oracle import layout as ol

pytestmark = pytest.mark.gpu

SMALL = [
    # lens, zigzag, causal
    ((100, 150, 130, 132), False, False),
    ((100, 150, 130, 132), False, True),
    ((1, 7, 64, 129), False, True),
    ((300,), False, False),
    ((300,), False, True),
    ((2, 6, 250, 32), True, True),
    ((128, 128, 128, 128), True, True),
    ((192, 64, 320, 128), True, False),
    ((66, 2, 130), True, True),
    ((512, 256, 768, 512), True, True),
]


def test_tiny_fp32_workload_forward():
    wl = WORKLOADS["tiny_fp32"]
    check_full(wl, run_case(wl, backward=False), backward=False)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("lens,zigzag,causal", SMALL)
def test_small_layouts_forward(lens, zigzag, causal, d, dtype):
    wl = Workload("small", B=2, H=2, d=d, lens=lens, causal=causal, zigzag=zigzag, dtype=dtype)
    check_full(wl, run_case(wl, seed=sum(lens) + d, backward=False), backward=False)


def test_vit1024_workload_forward_full():
    wl = WORKLOADS["vit1024_s4096"]
    check_full(wl, run_case(wl, backward=False), backward=False)


def test_scale_argument():
    for dtype in ("f32", "bf16"):
        wl = Workload("scale", B=1, H=2, d=64, lens=(96, 160), causal=True, zigzag=False, dtype=dtype)
        q, k, v = (x.cuda() for x in make_inputs(wl, seed=5))
        lay = st.Layout(wl.lens)
        out, lse = st.st_attn_fwd(lay, q, k, v, causal=True, scale=0.3)
        ro, rl = oa.forward(f64(q), f64(k), f64(v), wl.lens, False, True, scale=0.3)
        assert_close(f64(out), ro, dtype, "out")
        assert_close(f64(lse), rl, dtype, "lse")


def test_repeated_calls_are_identical():
    wl = Workload("rep", B=1, H=4, d=128, lens=(1024, 512, 512), causal=True, zigzag=True, dtype="bf16")
    q, k, v = (x.cuda() for x in make_inputs(wl, seed=9))
    lay = st.Layout(wl.lens, True)
    o1, l1 = st.st_attn_fwd(lay, q, k, v, causal=True)
    o2, l2 = st.st_attn_fwd(lay, q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# ------------------------------------------------------------- partials, merge, permute

PARTIAL_LAYOUTS = [
    ((100, 150, 130, 132), False, False),
    ((2, 6, 250, 32), True, True),
    ((128, 128, 128, 128), True, True),
    ((512, 256, 768, 512), True, True),
    ((300,), False, True),
    ((256, 256, 256, 256), False, False),     # every tile full
    ((1, 7, 64, 129), False, True),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("lens,zigzag,causal", PARTIAL_LAYOUTS)
def test_partials_match_oracle_and_merge_to_attention(lens, zigzag, causal, d, dtype):
    """The partials mode (bf16: the tensor-core forward writing and restarting its state at every KV shard)
    against the oracle's per-(query row, KV shard) partials, and the standalone merge of those partials
    against the oracle's full attention."""
    wl = Workload("part", B=2, H=2, d=d, lens=lens, causal=causal, zigzag=zigzag, dtype=dtype)
    q, k, v = (x.cuda() for x in make_inputs(wl, seed=11 + d))
    lay = st.Layout(lens, zigzag)
    po, pl = st.st_attn_fwd_partials(lay, q, k, v, causal=causal)
    torch.cuda.synchronize()
    assert_no_device_error()
    Q, K, V = f64(q), f64(k), f64(v)
    ro, rl = oa.ring_partials(Q, K, V, lens, zigzag, causal)
    assert_close(f64(po), ro, dtype, "partial_out")
    assert_lse(f64(pl), rl, dtype, "partial_lse")
    mo, ml = st.st_attn_merge(po, pl, out_dtype=torch.float32)
    torch.cuda.synchronize()
    fo, fl = oa.forward(Q, K, V, lens, zigzag, causal)
    assert_close(f64(mo), fo, dtype, "merged out")
    assert_lse(f64(ml), fl, dtype, "merged lse")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_merge_kernel_against_oracle(d, out_dtype):
    D, B, S, H = 5, 2, 77, 3
    g = torch.Generator().manual_seed(7)
    po = torch.randn(D, B, S, H, d, generator=g)
    pl = torch.randn(D, B, H, S, generator=g) * 3
    pl[1] = -float("inf")                       # an empty partial
    pl[:, 0, 0, 5] = -float("inf")              # a row with no visible key at all
    mo, ml = st.st_attn_merge(po.cuda(), pl.cuda(), out_dtype=out_dtype)
    torch.cuda.synchronize()
    ro, rl = oa.merge_partials(po.double().numpy(), pl.double().numpy().transpose(0, 1, 3, 2))
    dt = "f32" if out_dtype == torch.float32 else "bf16"
    assert_close(f64(mo), ro, dt, "merge out")
    assert_lse(f64(ml), rl.transpose(0, 2, 1), dt, "merge lse")


@pytest.mark.parametrize("lens,zigzag", [((100, 150, 130, 132), False), ((2, 6, 250, 32), True),
                                         ((12928, 19392, 384, 64), True)])
def test_permute_round_trip(lens, zigzag):
    S = sum(lens)
    x = torch.randn(2, S, 3, 64, dtype=torch.bfloat16, device="cuda")
    lay = st.Layout(lens, zigzag)
    nat = st.st_permute(lay, x, to_natural=True)
    back = st.st_permute(lay, nat, to_natural=False)
    torch.cuda.synchronize()
    pos = ol.natural_positions(list(lens), zigzag)
    ref = np.empty_like(f64(x))
    ref[:, pos] = f64(x)
    assert np.array_equal(f64(nat), ref)
    assert torch.equal(back, x)


# ------------------------------------------------------------- full-size workloads

@pytest.mark.slow
def test_vit4096_workload_sampled_rows():
    """The ViT 4096^2 workload at full size: 192 sampled rows of three heads, and every one of the
    65536 rows of head 7 (out and lse) against the oracle."""
    import os
    wl = WORKLOADS["vit4096_s65536"]
    res = run_case(wl, backward=False)
    rows = sample_rows(wl.S, 192, seed=3)
    check_rows(wl, res, rows, [(0, 0), (0, 7), (0, 15)])
    h = 7
    Q, K, V = (f64(x[0:1, :, h:h + 1]) for x in res["in"][:3])
    outs, lses, _ = oa.row_stats(Q, K, V, np.zeros_like(Q), wl.lens, wl.zigzag, wl.causal,
                                 workers=max(1, min(16, os.cpu_count() or 1)))
    assert_close(f64(res["out"][0, :, h]), outs[(0, 0)], wl.dtype, "out[0,7] (all rows)")
    assert_close(f64(res["lse"][0, h]), lses[(0, 0)], wl.dtype, "lse[0,7] (all rows)")


@pytest.mark.slow
def test_llm7b_causal_workload_sampled_rows():
    wl = WORKLOADS["llm7b_causal_s131072"]
    res = run_case(wl, backward=False)
    pos = ol.natural_positions(list(wl.lens), wl.zigzag)
    # the first natural rows (few keys) and rows at chunk edges
    edges = [int(np.where(pos == p)[0][0]) for p in (0, 1, 2, 127, 128, 8191, 8192, 131071)]
    rows = np.unique(np.concatenate([sample_rows(wl.S, 96, seed=4), edges]))
    check_rows(wl, res, rows, [(0, 0), (0, 31)])


@pytest.mark.slow
def test_train_workload_forward_sampled_rows():
    wl = WORKLOADS["train_s32768"]
    res = run_case(wl, backward=False)
    pos = ol.natural_positions(list(wl.lens), wl.zigzag)
    edges = [int(np.where(pos == p)[0][0]) for p in (0, 1, 6463, 6464, 32767)]
    rows = np.unique(np.concatenate([sample_rows(wl.S, 96, seed=5), edges]))
    check_rows(wl, res, rows, [(0, 0), (1, 31)])
