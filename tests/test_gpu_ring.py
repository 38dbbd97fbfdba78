"""GPU parity of ring attention across ranks (ShardTensor summary, section 4, ring attention), through the C-ABI.

Rank r keeps the queries of shard r; the K/V shards travel round the ring (in training with their dK/dV
accumulators).  Here the D ranks are held on one GPU (st_ring_fwd_local / st_ring_bwd_local: every rank's
buffers apart, the blocks passed by device-to-device copies on a second stream while the previous blocks
compute), and one step of one rank is also called alone (st_ring_fwd_step / st_ring_bwd_step).  Everything is
held to the float64 oracle with the bf16 bounds.
"""
import numpy as np
import pytest
import torch

import domain_ring_attention_gb300 as st
from domain_ring_attention_gb300 import _lib
from domain_ring_attention_gb300.workloads import Workload, make_inputs
from gpu_common import assert_close, assert_lse, assert_no_device_error, f64
from oracle import attention as oa
from oracle import layout as ol

pytestmark = pytest.mark.gpu

LAYOUTS = [
    ((100, 150, 130, 132), False, False),
    ((512, 256, 768, 512), True, True),
    ((2, 6, 250, 32), True, True),
    ((256, 256), False, True),
    ((384, 128, 640), False, False),
    ((300,), False, True),
    ((640, 128, 2, 384, 256, 512, 64, 96), True, True),     # eight ranks, uneven, a 2-row shard
]


def shards(x, lens):
    off = ol.shard_offsets(list(lens))
    return [x[:, off[r]:off[r + 1]].contiguous() for r in range(len(lens))]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("lens,zigzag,causal", LAYOUTS)
def test_ring_forward_and_backward_on_one_gpu(lens, zigzag, causal, d):
    wl = Workload("ring", B=2, H=2, d=d, lens=lens, causal=causal, zigzag=zigzag, dtype="bf16")
    q, k, v, do = (x.cuda() for x in make_inputs(wl, seed=31 + d, with_dout=True))
    lay = st.Layout(lens, zigzag)
    qs, ks, vs, dos = (shards(x, lens) for x in (q, k, v, do))
    outs, lses = _lib.st_ring_fwd_local(lay, qs, ks, vs, causal=causal, out_dtype=torch.float32)
    outs16, lses16 = _lib.st_ring_fwd_local(lay, qs, ks, vs, causal=causal, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert_no_device_error()
    Q, K, V, DO = (f64(x) for x in (q, k, v, do))
    ro, rl = oa.forward(Q, K, V, lens, zigzag, causal)
    off = ol.shard_offsets(list(lens))
    for r in range(len(lens)):
        rows = slice(off[r], off[r + 1])
        assert_close(f64(outs[r]), ro[:, rows], "bf16", "out of rank %d" % r)
        assert_lse(f64(lses[r]), rl[:, :, rows], "bf16", "lse of rank %d" % r)
        # the bf16 output of the last step is the merged fp32 value rounded once
        assert torch.equal(outs16[r], outs[r].to(torch.bfloat16))
        assert torch.equal(lses16[r], lses[r])
    dqs, dks, dvs = _lib.st_ring_bwd_local(lay, qs, ks, vs, outs, lses, dos, causal=causal)
    torch.cuda.synchronize()
    assert_no_device_error()
    gq, gk, gv = oa.backward(Q, K, V, ro, rl, DO, lens, zigzag, causal)
    for name, got, ref in (("dq", dqs, gq), ("dk", dks, gk), ("dv", dvs, gv)):
        full = np.concatenate([f64(x) for x in got], axis=1)
        assert_close(full, ref, "bf16", name, rel_rms=True)


@pytest.mark.parametrize("lens,zigzag,causal", [((512, 256, 768, 512), True, True), ((100, 150, 130, 132), False, False)])
def test_ring_steps_of_one_rank(lens, zigzag, causal):
    """One rank's steps called alone: the first step's output is its block's partial (the oracle's
    partial_block), and folding the remaining blocks in ring order gives the rank's rows of attention."""
    d = 128
    wl = Workload("step", B=1, H=2, d=d, lens=lens, causal=causal, zigzag=zigzag, dtype="bf16")
    q, k, v = (x.cuda() for x in make_inputs(wl, seed=41))
    lay = st.Layout(lens, zigzag)
    qs, ks, vs = (shards(x, lens) for x in (q, k, v))
    Q, K, V = (f64(x) for x in (q, k, v))
    pos = ol.natural_positions(list(lens), zigzag)
    off = ol.shard_offsets(list(lens))
    D = len(lens)
    r = D - 1
    rows = slice(off[r], off[r + 1])
    state = None
    for t in range(D):
        j = (r - t) % D
        out, lse = _lib.st_ring_fwd_step(lay, r, j, qs[r], ks[j], vs[j], prev=state, causal=causal,
                                         out=None if state is None else state[0],
                                         lse=None if state is None else state[1])
        if t == 0:
            torch.cuda.synchronize()
            kr = slice(off[j], off[j + 1])
            for h in range(2):
                po, pl = oa.partial_block(Q[0, rows, h], K[0, kr, h], V[0, kr, h], pos[rows], pos[kr], causal,
                                          1 / np.sqrt(d))
                assert_close(f64(out[0, :, h]), po, "bf16", "first-step partial")
                assert_lse(f64(lse[0, h]), pl, "bf16", "first-step partial lse")
        state = (out, lse)
    torch.cuda.synchronize()
    assert_no_device_error()
    ro, rl = oa.forward(Q, K, V, lens, zigzag, causal)
    assert_close(f64(state[0]), ro[:, rows], "bf16", "rank rows after the ring")
    assert_lse(f64(state[1]), rl[:, :, rows], "bf16", "rank lse after the ring")


@pytest.mark.slow
def test_ring_on_the_7b_layout_sampled():
    """The 7B-style layout (8 ranks, 16 zigzag chunks, causal) at S = 131072 with 2 heads: the ring forward
    on one GPU, every rank's first and last rows, its chunk edges and a random sample against the oracle."""
    lens = (16384,) * 8
    wl = Workload("ring7b", B=1, H=2, d=128, lens=lens, causal=True, zigzag=True, dtype="bf16")
    q, k, v = make_inputs(wl, seed=5, device=torch.device("cuda"))
    lay = st.Layout(lens, True)
    qs, ks, vs = (shards(x, lens) for x in (q, k, v))
    outs, lses = _lib.st_ring_fwd_local(lay, qs, ks, vs, causal=True, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert_no_device_error()
    off = ol.shard_offsets(list(lens))
    rng = np.random.default_rng(3)
    local = np.unique(np.concatenate([[0, 8191, 8192, 16383], rng.choice(16384, 12, replace=False)]))
    rows = np.concatenate([off[r] + local for r in range(8)])
    Q, K, V = (f64(x) for x in (q, k, v))
    ro, rl = oa.forward_rows(Q, K, V, lens, True, True, rows)
    got_o = np.concatenate([f64(outs[r][:, torch.as_tensor(local, device="cuda")]) for r in range(8)], axis=1)
    got_l = np.concatenate([f64(lses[r][:, :, torch.as_tensor(local, device="cuda")]) for r in range(8)], axis=2)
    for h in range(2):
        assert_close(got_o[0, :, h], ro[(0, h)], "bf16", "out head %d" % h)
        assert_close(got_l[0, h], rl[(0, h)], "bf16", "lse head %d" % h)
