"""GPU checks of the host-buffer forward (st_attn_fwd_host).

It must give, bit for bit, what st_attn_fwd gives on the same inputs: the same kernels on the same tiles, only
launched per group of heads (or per chunk of query tiles) with the copies overlapped.  With head groups the fp16
copy of V is scaled per group, by another power of two than the whole tensor's; the products and the final
normalisation then differ by exact powers of two only, so the outputs are still the same bits.  The cases:
- one chunk (few tiles, H = 4: no head groups);
- head groups of 1, 16, 14 and 1 heads (B * H * tiles large enough for groups of 16);
- head groups of 1, 4, 4, 4, 2 and 1 heads;
- causal zigzag over uneven shards in head groups of 1, 16, 14 and 1 (heaviest tiles first within each group);
- three chunks of query tiles (H = 3 has no divisor that leaves four waves per group);
- head groups of uneven sizes (1, 3, 1, 1 for H = 6; 1, 3, 2, 1 for H = 7, which has no divisor);
- causal zigzag at d = 64 in head groups of 1, 2, 2, 2, 1.
A few rows are also held to the oracle with the bf16 bounds.
"""
import numpy as np
import pytest
import torch

import domain_ring_attention_gb300 as st
from domain_ring_attention_gb300.workloads import Workload, make_inputs
from oracle import attention as oa
from gpu_common import assert_no_device_error, f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H,d,lens,causal,zigzag", [
    (1, 4, 64, (512,) * 8, False, False),              # one chunk
    (2, 32, 64, (1024,) * 8, False, False),            # head groups of 1, 16, 14, 1
    (2, 16, 64, (2432,) * 8, False, False),            # head groups of 1, 4, 4, 4, 2, 1 (80 tiles x 2 CTAs per head)
    (2, 32, 128, (2560, 1536, 3328, 768), True, True),  # head groups of 1, 16, 14, 1; causal zigzag, uneven shards
    (2, 3, 64, (8192,) * 8, False, False),             # three chunks of query tiles: 51 + 154 + 51
    (1, 6, 64, (16384,) * 4, False, False),            # head groups of 1, 3, 1, 1
    (2, 8, 64, (12288, 20480, 4096, 2048), True, True),  # head groups of 1, 2, 2, 2, 1; causal zigzag, d = 64
    (1, 7, 128, (8192,) * 8, False, False),            # H = 7 (no divisor): head groups of 1, 3, 2, 1
])
def test_host_forward_equals_device_forward(B, H, d, lens, causal, zigzag):
    wl = Workload("host", B=B, H=H, d=d, lens=lens, causal=causal, zigzag=zigzag, dtype="bf16")
    q, k, v = make_inputs(wl, seed=3)
    lay = st.Layout(lens, zigzag=zigzag)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    ref_out, ref_lse = st.st_attn_fwd(lay, qd, kd, vd, causal=causal)
    pin = [x.pin_memory() for x in (q, k, v)]
    out_h = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=True)
    lse_h = torch.empty(tuple(ref_lse.shape), dtype=torch.float32, pin_memory=True)
    dev = {"q": torch.empty_like(qd), "k": torch.empty_like(kd), "v": torch.empty_like(vd),
           "out": torch.empty_like(qd), "lse": torch.empty_like(ref_lse)}
    st.st_attn_fwd_host(lay, pin[0], pin[1], pin[2], out_h, lse_h, dev, causal=causal)
    torch.cuda.current_stream().synchronize()
    assert_no_device_error()
    assert torch.equal(out_h, ref_out.cpu())
    assert torch.equal(lse_h, ref_lse.cpu())
    # a few rows against the oracle: the first query row of every shard, for head 0 of batch 0
    rows = np.cumsum((0,) + lens[:-1])
    outs, lses = oa.forward_rows(f64(q), f64(k), f64(v), lens, zigzag, causal, rows, heads=[(0, 0)])
    o, l = outs[(0, 0)], lses[(0, 0)]
    err = np.abs(f64(out_h[0, rows, 0]) - o)
    assert err.max() <= 1e-2, err.max()
    assert np.abs(f64(lse_h[0, 0, rows]) - l).max() <= 1e-2


def test_host_forward_waits_for_work_already_queued_on_its_stream():
    """The copies run on a second stream, but only after the work queued on `stream` before the call: here
    `stream` first spins (~25 ms) and then overwrites the device staging buffer of v.  A copy that started at
    once would be overwritten by that late write; the call must instead copy v in after it, and give the outputs
    of st_attn_fwd bit for bit."""
    wl = Workload("order", B=1, H=4, d=64, lens=(512,) * 8, causal=False, zigzag=False, dtype="bf16")
    q, k, v = make_inputs(wl, seed=5)
    lay = st.Layout(wl.lens)
    ref_out, ref_lse = st.st_attn_fwd(lay, q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    pin = [x.pin_memory() for x in (q, k, v)]
    out_h = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=True)
    lse_h = torch.empty(tuple(ref_lse.shape), dtype=torch.float32, pin_memory=True)
    dev = {"q": torch.empty_like(ref_out), "k": torch.empty_like(ref_out), "v": torch.empty_like(ref_out),
           "out": torch.empty_like(ref_out), "lse": torch.empty_like(ref_lse)}
    stream, copy_stream = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(stream):
        torch.cuda._sleep(50_000_000)
        dev["v"].fill_(7.0)
    st.st_attn_fwd_host(lay, pin[0], pin[1], pin[2], out_h, lse_h, dev, stream=stream, copy_stream=copy_stream)
    stream.synchronize()
    assert_no_device_error()
    assert torch.equal(out_h, ref_out.cpu())
    assert torch.equal(lse_h, ref_lse.cpu())
