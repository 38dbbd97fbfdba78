"""GPU parity: the CUDA library (through the C-ABI) against the float64 oracle.

Tolerances (stated for this method): fp32 inputs -- max abs error <= 1e-5;
bf16 inputs with fp32 accumulation -- max abs <= 1e-2 and mean abs <= 1e-3.
Gradients use the same bounds relative to the RMS of the oracle gradient.
Small cases are compared element by element; the full-size workloads are
compared on sampled rows (rows are independent, so each sampled row is exact)
and, for the backward, on whole sampled heads.
"""
import numpy as np
import pytest
import torch

import domain_ring_attention_gb300 as st
from domain_ring_attention_gb300.workloads import WORKLOADS, Workload, make_inputs, sample_rows
from oracle import attention as oa
from oracle import layout as ol

pytestmark = pytest.mark.gpu


def f64(t):
    return t.detach().float().cpu().double().numpy()


def assert_close(got, ref, dtype, name, rel_rms=False):
    err = np.abs(np.asarray(got, dtype=np.float64) - ref)
    den = float(np.sqrt(np.mean(ref * ref))) if rel_rms else 1.0
    mx, mean = err.max() / den, err.mean() / den
    if dtype == "f32":
        assert mx <= 1e-5, "%s: max err %.3e > 1e-5" % (name, mx)
    else:
        assert mx <= 1e-2 and mean <= 1e-3, "%s: max %.3e mean %.3e" % (name, mx, mean)
    return mx, mean


def assert_lse(got, ref, dtype, name="lse"):
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), name + ": -inf pattern differs"
    assert_close(got[fin], ref[fin], dtype, name)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available()
    st.load()


def run_case(wl, seed=0, backward=True, grad_dtype=torch.float32):
    q, k, v, do = (x.cuda() for x in make_inputs(wl, seed=seed, with_dout=True))
    lay = st.Layout(wl.lens, wl.zigzag)
    out, lse = st.st_attn_fwd(lay, q, k, v, causal=wl.causal)
    res = {"out": out, "lse": lse, "in": (q, k, v, do)}
    if backward:
        res["grads"] = st.st_attn_bwd(lay, q, k, v, out, lse, do, causal=wl.causal,
                                      grad_dtype=grad_dtype)
    torch.cuda.synchronize()
    return res


def check_full(wl, res, backward=True):
    q, k, v, do = (f64(x) for x in res["in"])
    ro, rl = oa.forward(q, k, v, wl.lens, wl.zigzag, wl.causal)
    assert_close(f64(res["out"]), ro, wl.dtype, "out")
    assert_lse(f64(res["lse"]), rl, wl.dtype)
    if backward:
        rg = oa.backward(q, k, v, ro, rl, do, wl.lens, wl.zigzag, wl.causal)
        for name, g, r in zip(("dq", "dk", "dv"), res["grads"], rg):
            assert_close(f64(g), r, wl.dtype, name, rel_rms=True)


# ------------------------------------------------------------- small, full compare

def test_tiny_fp32_workload():
    wl = WORKLOADS["tiny_fp32"]
    check_full(wl, run_case(wl))


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
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("lens,zigzag,causal", SMALL)
def test_small_layouts(lens, zigzag, causal, d, dtype):
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


def test_vit1024_workload_full():
    wl = WORKLOADS["vit1024_s4096"]
    check_full(wl, run_case(wl), backward=True)


def test_scale_argument():
    wl = Workload("scale", B=1, H=2, d=64, lens=(96, 160), causal=True, zigzag=False, dtype="f32")
    q, k, v = (x.cuda() for x in make_inputs(wl, seed=5))
    lay = st.Layout(wl.lens)
    out, lse = st.st_attn_fwd(lay, q, k, v, causal=True, scale=0.3)
    ro, rl = oa.forward(f64(q), f64(k), f64(v), wl.lens, False, True, scale=0.3)
    assert_close(f64(out), ro, "f32", "out")
    assert_close(f64(lse), rl, "f32", "lse")


# ------------------------------------------------------------- partials, merge, permute

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("lens,zigzag,causal", [((100, 150, 130, 132), False, False),
                                                ((2, 6, 250, 32), True, True),
                                                ((128, 128, 128, 128), True, True)])
def test_partials_match_oracle_and_merge_to_fused(lens, zigzag, causal, dtype):
    wl = Workload("part", B=2, H=2, d=64, lens=lens, causal=causal, zigzag=zigzag, dtype=dtype)
    q, k, v = (x.cuda() for x in make_inputs(wl, seed=11))
    lay = st.Layout(lens, zigzag)
    po, pl = st.st_attn_fwd_partials(lay, q, k, v, causal=causal)
    ro, rl = oa.ring_partials(f64(q), f64(k), f64(v), lens, zigzag, causal)
    assert_close(f64(po), ro, "f32" if dtype == "f32" else "bf16", "partial_out")
    assert_lse(f64(pl), rl, dtype, "partial_lse")
    mo, ml = st.st_attn_merge(po, pl, out_dtype=q.dtype)
    fo, fl = st.st_attn_fwd(lay, q, k, v, causal=causal)
    torch.cuda.synchronize()
    fo64, ml64 = f64(fo), f64(ml)
    assert_close(f64(mo), fo64, dtype, "merged vs fused")
    assert_close(ml64, f64(fl), dtype, "merged lse vs fused")


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

def check_rows(wl, res, rows, heads):
    qd, kd, vd = res["in"][:3]
    out, lse = f64(res["out"]), f64(res["lse"])
    errs = []
    for (b, h) in heads:
        qh = f64(qd[b:b + 1, :, h:h + 1])
        kh = f64(kd[b:b + 1, :, h:h + 1])
        vh = f64(vd[b:b + 1, :, h:h + 1])
        ro, rl = oa.forward_rows(qh, kh, vh, wl.lens, wl.zigzag, wl.causal, rows, heads=[(0, 0)])
        errs.append(assert_close(out[b, rows, h], ro[(0, 0)], wl.dtype, "out[%d,%d]" % (b, h)))
        assert_close(lse[b, h, rows], rl[(0, 0)], wl.dtype, "lse[%d,%d]" % (b, h))
    return errs


@pytest.mark.slow
def test_vit4096_workload_sampled_rows():
    wl = WORKLOADS["vit4096_s65536"]
    res = run_case(wl, backward=False)
    rows = sample_rows(wl.S, 192, seed=3)
    check_rows(wl, res, rows, [(0, 0), (0, 7), (0, 15)])


@pytest.mark.slow
def test_llm7b_causal_workload_sampled_rows():
    wl = WORKLOADS["llm7b_causal_s131072"]
    res = run_case(wl, backward=False)
    pos = ol.natural_positions(list(wl.lens), wl.zigzag)
    # include the first natural rows (few keys) and rows at every chunk edge
    edges = [int(np.where(pos == p)[0][0]) for p in (0, 1, 2, 127, 128, 8191, 8192, 131071)]
    rows = np.unique(np.concatenate([sample_rows(wl.S, 96, seed=4), edges]))
    check_rows(wl, res, rows, [(0, 0), (0, 31)])


@pytest.mark.slow
def test_train_workload_fwd_rows_and_bwd_head():
    wl = WORKLOADS["train_s32768"]
    res = run_case(wl, backward=True)
    rows = sample_rows(wl.S, 96, seed=5)
    check_rows(wl, res, rows, [(0, 0), (1, 31)])
    # one whole head through the float64 backward
    b, h = 1, 5
    q, k, v, do = (f64(x[b:b + 1, :, h:h + 1]) for x in res["in"])
    ro, rl = oa.forward(q, k, v, wl.lens, wl.zigzag, wl.causal)
    rg = oa.backward(q, k, v, ro, rl, do, wl.lens, wl.zigzag, wl.causal)
    for name, g, r in zip(("dq", "dk", "dv"), res["grads"], rg):
        assert_close(f64(g[b:b + 1, :, h:h + 1]), r, wl.dtype, name, rel_rms=True)
