"""GPU parity of the backward path against the float64 oracle, through the C-ABI."""
import numpy as np
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


def half_ulp_bf16(x):
    """Half the spacing of bf16 numbers at each value of x (0 at 0): the most that rounding a real
    number to the bf16 value x can have moved it."""
    m, e = np.frexp(np.abs(x))              # |x| = m 2^e, m in [0.5, 1): spacing 2^(e - 8)
    return np.where(x == 0, 0.0, np.ldexp(1.0, e - 9))


@pytest.mark.parametrize("d", [64, 128])
def test_backward_determinism_and_bf16_gradients(d):
    """Two backward runs and a bf16-gradient run of the same case, all held to the oracle.

    dK and dV of a key tile are accumulated by one CTA, query tile after query tile in a fixed order, so they
    are bitwise reproducible, and the bf16 ones are the fp32 ones rounded once (with fewer than 8 query tiles
    per key tile, as here, the fp32 path takes no intermediate sums either).  dQ is added into an fp32
    accumulator by TMA reductions from the CTAs of all key tiles, in an order that varies from run to run, so
    it is not bitwise reproducible: its bf16 value is compared with the oracle, allowing half a bf16 spacing
    on top of the fp32 bound.  At d = 64 two threads issue the MMAs (dK by either, ordered through barriers),
    and with bf16 gradients the dQ drain runs one tile late; neither may change dK or dV by a bit."""
    wl = Workload("small", B=1, H=3, d=d, lens=(256, 128, 384), causal=True, zigzag=True, dtype="bf16")
    res_a = run_case(wl, seed=3)
    res_b = run_case(wl, seed=3)
    res16 = run_case(wl, seed=3, grad_dtype=torch.bfloat16)
    check_full(wl, res_a)                                  # fp32 gradients against the oracle
    check_full(wl, res_b)
    (dq_a, dk_a, dv_a), (dq_b, dk_b, dv_b) = res_a["grads"], res_b["grads"]
    dq16, dk16, dv16 = res16["grads"]
    assert dq16.dtype == dk16.dtype == dv16.dtype == torch.bfloat16
    assert torch.equal(dk_a, dk_b) and torch.equal(dv_a, dv_b)
    assert torch.equal(dk16, dk_a.to(torch.bfloat16))
    assert torch.equal(dv16, dv_a.to(torch.bfloat16))
    q, k, v, do = (f64(x) for x in res16["in"])
    ro, rl = oa.forward(q, k, v, wl.lens, wl.zigzag, wl.causal)
    rq = oa.backward(q, k, v, ro, rl, do, wl.lens, wl.zigzag, wl.causal)[0]
    got = f64(dq16)
    rms = float(np.sqrt(np.mean(rq * rq)))
    excess = np.maximum(np.abs(got - rq) - half_ulp_bf16(got), 0.0) / rms
    assert excess.max() <= 1e-2 and excess.mean() <= 1e-3, (excess.max(), excess.mean())


def test_d64_causal_bf16_gradients_many_tiles():
    """d = 64, causal zigzag over uneven shards, bf16 gradients, 24 query tiles per key tile.

    This covers the d = 64 schedule where the dQ drain of a tile runs after the next tile's softmax pass.
    With bf16 gradients the lead key tile has no intermediate fp32 flushes, and it is split into hi + lo
    parts on every tile, so dK and the next dP^T are issued by the first thread there.  All three gradients
    are held to the oracle at the fp32 bound plus half a bf16 spacing."""
    wl = Workload("d64long", B=1, H=2, d=64, lens=(1536, 1024, 512), causal=True, zigzag=True, dtype="bf16")
    res = run_case(wl, seed=8, grad_dtype=torch.bfloat16)
    q, k, v, do = (f64(x) for x in res["in"])
    ro, rl = oa.forward(q, k, v, wl.lens, wl.zigzag, wl.causal)
    ref = oa.backward(q, k, v, ro, rl, do, wl.lens, wl.zigzag, wl.causal)
    for name, g, r in zip(("dq", "dk", "dv"), res["grads"], ref):
        assert g.dtype == torch.bfloat16
        got = f64(g)
        rms = float(np.sqrt(np.mean(r * r)))
        excess = np.maximum(np.abs(got - r) - half_ulp_bf16(got), 0.0) / rms
        assert excess.max() <= 1e-2 and excess.mean() <= 1e-3, (name, excess.max(), excess.mean())


@pytest.mark.parametrize("d,causal,dtype", [(64, False, "f32"), (64, True, "bf16"), (128, False, "bf16"),
                                             (128, True, "bf16")])
def test_single_token_sequence(d, causal, dtype):
    """The degenerate layout: one shard of one token (S = 1).  out = v and lse is the one score; the softmax
    over a single key is constant, so dS = 0, the exact dQ and dK are zero and dV = dO.  dQ and dK are held to
    the bound on the scale of dV, since their own RMS is zero."""
    wl = Workload("one_token", B=2, H=3, d=d, lens=(1,), causal=causal, zigzag=False, dtype=dtype)
    res = run_case(wl, seed=5)
    check_full(wl, res)
    q, k, v, do = (f64(x) for x in res["in"])
    assert np.array_equal(f64(res["out"]), v), "out is not v"


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
    """The training workload at full size: every gradient element of head (1, 5) against the oracle's full
    backward, and for head (0, 0) every forward row plus sampled dQ rows and dK / dV key columns (the lead
    tile, the shard and chunk edges, 256 random) against the oracle's row statistics."""
    import os
    from oracle import layout as ol
    wl = WORKLOADS["train_s32768"]
    res = run_case(wl, backward=True)
    b, h = 1, 5
    q, k, v, do = (f64(x[b:b + 1, :, h:h + 1]) for x in res["in"])
    ro, rl = oa.forward(q, k, v, wl.lens, wl.zigzag, wl.causal)
    rg = oa.backward(q, k, v, ro, rl, do, wl.lens, wl.zigzag, wl.causal)
    for name, g, r in zip(("dq", "dk", "dv"), res["grads"], rg):
        assert_close(f64(g[b:b + 1, :, h:h + 1]), r, wl.dtype, name, rel_rms=True)
    b, h = 0, 0
    S = wl.S
    Q, K, V, DO = (f64(x[b:b + 1, :, h:h + 1]) for x in res["in"])
    outs, lses, deltas = oa.row_stats(Q, K, V, DO, wl.lens, wl.zigzag, True,
                                      workers=max(1, min(16, os.cpu_count() or 1)))
    assert_close(f64(res["out"][b, :, h]), outs[(0, 0)], "bf16", "out[0,0] (all rows)")
    pos = ol.natural_positions(list(wl.lens), wl.zigzag)
    at = np.argsort(pos)
    lead = at[:128]
    rest = np.setdiff1d(np.arange(S), lead)
    sample = np.sort(np.random.default_rng(11).choice(rest, size=256, replace=False))
    off = ol.shard_offsets(list(wl.lens))
    mids = [off[r] + wl.lens[r] // 2 for r in range(len(wl.lens))]          # zigzag chunk boundaries
    edges = np.unique(np.concatenate([[o, o - 1] for o in list(off[1:-1]) + mids] + [[0, S - 1]]))
    dq, dk, dv = res["grads"]
    pick = lambda t, idx: f64(t[b, torch.as_tensor(idx, device=t.device), h])
    rows = np.concatenate([lead, sample])
    rq = oa.backward_rows(Q, K, V, DO, wl.lens, wl.zigzag, True, np.concatenate([rows, edges]),
                          heads=[(0, 0)])[(0, 0)]
    _stratified_check(pick(dq, rows), rq[:len(rows)], 128, S, "dq[0,0]", pick(dq, edges), rq[len(rows):])
    rk, rv = oa.backward_cols(Q, K, V, DO, wl.lens, wl.zigzag, True, np.concatenate([rows, edges]), lses, deltas)
    _stratified_check(pick(dk, rows), rk[(0, 0)][:len(rows)], 128, S, "dk[0,0]", pick(dk, edges),
                      rk[(0, 0)][len(rows):])
    _stratified_check(pick(dv, rows), rv[(0, 0)][:len(rows)], 128, S, "dv[0,0]", pick(dv, edges),
                      rv[(0, 0)][len(rows):])


def _stratified_check(got, ref, n_lead, n_total, name, extra_got=None, extra_ref=None):
    """Hold sampled gradient rows to the bf16 bounds relative to the RMS of the whole tensor.

    The first ``n_lead`` rows of ``ref`` are a whole stratum (e.g. every key of the lead tile), the rest a
    uniform random sample of the other ``n_total - n_lead`` rows, so the tensor's RMS and mean error are
    estimated without bias from the two strata.  ``extra_*`` rows (chunk edges) count toward the maximum."""
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(np.asarray(got, dtype=np.float64) - ref)
    w_rest = (n_total - n_lead) / max(1, len(ref) - n_lead)
    sq = (np.sum(ref[:n_lead] ** 2) + w_rest * np.sum(ref[n_lead:] ** 2)) / (n_total * ref.shape[1])
    rms = float(np.sqrt(sq))
    mean_err = (np.sum(err[:n_lead]) + w_rest * np.sum(err[n_lead:])) / (n_total * ref.shape[1])
    mx = err.max()
    if extra_got is not None:
        mx = max(mx, np.abs(np.asarray(extra_got, dtype=np.float64) - extra_ref).max())
    assert mx / rms <= 1e-2 and mean_err / rms <= 1e-3, "%s: max %.3e mean %.3e (of RMS %.3e)" % (
        name, mx / rms, mean_err / rms, rms)
    return mx / rms, mean_err / rms


@pytest.mark.slow
def test_llm7b_causal_workload_backward_sampled():
    """The 7B-style causal workload at full size (B1 H32 d128, S = 131072, D = 8 zigzag shards = 16 chunks
    of 8192): forward and backward through the C-ABI, held to the oracle on two heads.

    For each head the oracle computes out, lse and Delta of all 131072 rows (the forward is compared on
    every row).  dQ is compared on the 128 first natural rows, 256 random rows and the rows at chunk
    edges; dK and dV on the keys of the lead tile (natural positions 0-127, seen by every query: their
    gradients are the largest and their tensor-memory accumulation is promoted to fp32 every 8 query
    tiles), 256 random keys and the keys at chunk edges, from the oracle's own lse and Delta."""
    import os
    from oracle import layout as ol
    from domain_ring_attention_gb300.workloads import make_inputs
    from gpu_common import assert_no_device_error

    wl = WORKLOADS["llm7b_causal_s131072"]
    dev = torch.device("cuda")
    q, k, v, do = make_inputs(wl, seed=0, device=dev, with_dout=True)
    lay = st.Layout(wl.lens, wl.zigzag)
    out, lse = st.st_attn_fwd(lay, q, k, v, causal=True, out_dtype=torch.float32)
    dq, dk, dv = st.st_attn_bwd(lay, q, k, v, out, lse, do, causal=True)
    torch.cuda.synchronize()
    assert_no_device_error()
    S = wl.S
    pos = ol.natural_positions(list(wl.lens), wl.zigzag)
    at = np.argsort(pos)                                   # natural position -> buffer row
    rng = np.random.default_rng(7)
    lead = at[:128]
    rest = np.setdiff1d(np.arange(S), lead)
    edges = np.unique(at[[c + o for c in range(8192, S, 8192) for o in (-1, 0)]])
    workers = max(1, min(16, os.cpu_count() or 1))
    pick = lambda t, b, idx, h: f64(t[b, torch.as_tensor(idx, device=t.device), h])
    for (b, h) in [(0, 0), (0, 31)]:
        Q, K, V, DO = (f64(x[b:b + 1, :, h:h + 1]) for x in (q, k, v, do))
        outs, lses, deltas = oa.row_stats(Q, K, V, DO, wl.lens, wl.zigzag, True, workers=workers)
        assert_close(f64(out[b, :, h]), outs[(0, 0)], "bf16", "out[%d,%d] (all rows)" % (b, h))
        assert_close(f64(lse[b, h]), lses[(0, 0)], "bf16", "lse[%d,%d] (all rows)" % (b, h))
        sample = np.sort(rng.choice(rest, size=256, replace=False))
        rows = np.concatenate([lead, sample])
        rq = oa.backward_rows(Q, K, V, DO, wl.lens, wl.zigzag, True, np.concatenate([rows, edges]),
                              heads=[(0, 0)])[(0, 0)]
        _stratified_check(pick(dq, b, rows, h), rq[:len(rows)], 128, S, "dq[%d,%d]" % (b, h),
                          pick(dq, b, edges, h), rq[len(rows):])
        cols = np.concatenate([lead, sample])
        rk, rv = oa.backward_cols(Q, K, V, DO, wl.lens, wl.zigzag, True, np.concatenate([cols, edges]),
                                  lses, deltas)
        rk, rv = rk[(0, 0)], rv[(0, 0)]
        _stratified_check(pick(dk, b, cols, h), rk[:len(cols)], 128, S, "dk[%d,%d]" % (b, h),
                          pick(dk, b, edges, h), rk[len(cols):])
        _stratified_check(pick(dv, b, cols, h), rv[:len(cols)], 128, S, "dv[%d,%d]" % (b, h),
                          pick(dv, b, edges, h), rv[len(cols):])
