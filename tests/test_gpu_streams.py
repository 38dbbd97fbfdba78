"""The Python binding on a stream other than torch's current one.

A call that allocates its own workspace frees it when it returns, while its kernels may still be queued on the
call's stream.  The binding records such tensors on that stream, so the caching allocator cannot hand their memory
to work on the current stream in the meantime.  Here the call's stream first spins (~25 ms), and a buffer of the
workspace's size is allocated and filled on the current stream right after the call returns: had it received the
workspace's memory, the fill would overwrite the fp16 copy of v before the attention kernel reads it.
"""
import pytest
import torch

import domain_ring_attention_gb300 as st
from domain_ring_attention_gb300.workloads import Workload, make_inputs
from gpu_common import assert_no_device_error

pytestmark = pytest.mark.gpu


def test_forward_on_a_side_stream_keeps_its_workspace():
    wl = Workload("side", B=1, H=4, d=64, lens=(2048,) * 4, causal=False, zigzag=False, dtype="bf16")
    q, k, v = (x.cuda() for x in make_inputs(wl, seed=9))
    lay = st.Layout(wl.lens)
    ref_out, ref_lse = st.st_attn_fwd(lay, q, k, v)
    torch.cuda.synchronize()
    need = st.st_attn_workspace_size(lay, wl.B, wl.H, wl.d, torch.bfloat16, 0)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        torch.cuda._sleep(50_000_000)
    out, lse = st.st_attn_fwd(lay, q, k, v, stream=side)      # its workspace is freed on return
    junk = torch.empty(max(need, 1), device="cuda", dtype=torch.uint8)
    junk.fill_(0x7B)                                           # on the current stream, not behind the spin
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    assert_no_device_error()
    assert torch.equal(out, ref_out)
    assert torch.equal(lse, ref_lse)
