"""GPU parity on seeded random layouts: shard counts, uneven lengths (shards of one token, lengths that end inside a
128-row tile, zigzag halves), causal or not, d = 64 or 128, fp32 or bf16, several batches and heads.

Each case runs the forward and the backward through the C-ABI and compares every output and gradient element with
the float64 oracle at the stated bounds.  bf16 cases also run the host-buffer forward, which must give the device
forward's outputs bit for bit.  A second set of bf16 layouts runs ring attention with its D ranks held on one GPU
(every rank's shard in buffers of its own, the K/V blocks passed round the ring; ShardTensor summary, section 4,
ring attention) against the same oracle.  The layouts come from a fixed seed, so a failure names a reproducible
case.
"""
import numpy as np
import pytest
import torch

import domain_ring_attention_gb300 as st
from domain_ring_attention_gb300 import _lib
from domain_ring_attention_gb300.workloads import Workload, make_inputs
from gpu_common import assert_close, assert_lse, assert_no_device_error, check_full, f64, run_case
from oracle import attention as oa
from oracle import layout as ol

pytestmark = pytest.mark.gpu


def random_cases(n=40, seed=20261203):
    rng = np.random.RandomState(seed)
    cases = []
    for i in range(n):
        # odd cases: fewer, longer shards (several 128- and 256-row tiles per shard)
        D = int(rng.randint(1, 7)) if i % 2 == 0 else int(rng.randint(1, 5))
        top = 250 if i % 2 == 0 else 700
        zigzag = bool(rng.rand() < 0.5)
        causal = bool(rng.rand() < 0.6)
        if zigzag:
            lens = tuple(int(2 * rng.randint(1, top // 2 + 1)) for _ in range(D))   # even: two halves per shard
        else:
            lens = tuple(int(rng.randint(1, top + 1)) for _ in range(D))
        if i % 5 == 0:                                                      # a shard of one or two tokens
            lens = (2 if zigzag else 1,) + lens[1:]
        d = 64 if rng.rand() < 0.5 else 128
        dtype = "f32" if i % 4 == 3 else "bf16"
        B, H = int(rng.randint(1, 3)), int(rng.randint(1, 4))
        cases.append((i, B, H, d, lens, causal, zigzag, dtype))
    return cases


@pytest.mark.parametrize("i,B,H,d,lens,causal,zigzag,dtype", random_cases())
def test_random_layout_forward_backward(i, B, H, d, lens, causal, zigzag, dtype):
    wl = Workload("random%d" % i, B=B, H=H, d=d, lens=lens, causal=causal, zigzag=zigzag, dtype=dtype)
    res = run_case(wl, seed=1000 + i)
    check_full(wl, res)
    if dtype != "bf16":
        return
    # the host-buffer forward on the same inputs: the device forward's outputs, bit for bit
    q, k, v = make_inputs(wl, seed=1000 + i)
    lay = st.Layout(lens, zigzag=zigzag)
    pin = [x.pin_memory() for x in (q, k, v)]
    out_h = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=True)
    lse_h = torch.empty(tuple(res["lse"].shape), dtype=torch.float32, pin_memory=True)
    dev = {"q": torch.empty_like(res["out_native"]), "k": torch.empty_like(res["out_native"]),
           "v": torch.empty_like(res["out_native"]), "out": torch.empty_like(res["out_native"]),
           "lse": torch.empty_like(res["lse"])}
    st.st_attn_fwd_host(lay, pin[0], pin[1], pin[2], out_h, lse_h, dev, causal=causal)
    torch.cuda.current_stream().synchronize()
    assert_no_device_error()
    assert torch.equal(out_h, res["out_native"].cpu())
    assert torch.equal(lse_h, res["lse"].cpu())


def ring_cases(n=12, seed=20261204):
    rng = np.random.RandomState(seed)
    cases = []
    for i in range(n):
        D = int(rng.randint(1, 7))
        zigzag = bool(rng.rand() < 0.5)
        causal = bool(rng.rand() < 0.6)
        if zigzag:
            lens = tuple(int(2 * rng.randint(1, 201)) for _ in range(D))
        else:
            lens = tuple(int(rng.randint(1, 401)) for _ in range(D))
        d = 64 if rng.rand() < 0.5 else 128
        B, H = int(rng.randint(1, 3)), int(rng.randint(1, 3))
        cases.append((i, B, H, d, lens, causal, zigzag))
    return cases


@pytest.mark.parametrize("i,B,H,d,lens,causal,zigzag", ring_cases())
def test_random_layout_ring_on_one_gpu(i, B, H, d, lens, causal, zigzag):
    wl = Workload("ring%d" % i, B=B, H=H, d=d, lens=lens, causal=causal, zigzag=zigzag, dtype="bf16")
    q, k, v, do = (x.cuda() for x in make_inputs(wl, seed=2000 + i, with_dout=True))
    lay = st.Layout(lens, zigzag)
    off = ol.shard_offsets(list(lens))
    qs, ks, vs, dos = ([x[:, off[r]:off[r + 1]].contiguous() for r in range(len(lens))] for x in (q, k, v, do))
    outs, lses = _lib.st_ring_fwd_local(lay, qs, ks, vs, causal=causal, out_dtype=torch.float32)
    dqs, dks, dvs = _lib.st_ring_bwd_local(lay, qs, ks, vs, outs, lses, dos, causal=causal)
    torch.cuda.synchronize()
    assert_no_device_error()
    Q, K, V, DO = (f64(x) for x in (q, k, v, do))
    ro, rl = oa.forward(Q, K, V, lens, zigzag, causal)
    out = np.concatenate([f64(x) for x in outs], axis=1)
    lse = np.concatenate([f64(x) for x in lses], axis=2)
    assert_close(out, ro, "bf16", "out")
    assert_lse(lse, rl, "bf16")
    gq, gk, gv = oa.backward(Q, K, V, ro, rl, DO, lens, zigzag, causal)
    dv_rms = float(np.sqrt(np.mean(gv * gv)))
    for name, got, ref in (("dq", dqs, gq), ("dk", dks, gk), ("dv", dvs, gv)):
        assert_close(np.concatenate([f64(x) for x in got], axis=1), ref, "bf16", name, rel_rms=True, scale=dv_rms)
