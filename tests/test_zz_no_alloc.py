"""st_attn_fwd_noalloc: the forward for callers that cannot allocate.

Some callers cannot allocate device memory: they are handed only their input
and output buffers (an operator inside another runtime), or their memory is
fixed at start-up, or their critical path must not call a device allocator.
st_attn_fwd_noalloc serves them from a fixed array of device memory inside the
library instead of a caller workspace.  Here it is called through the C-ABI
and compared with st_attn_fwd on the same inputs, on two calls in a row with
different inputs (the shared array keeps the previous call's contents), and a
problem too large for the array must be refused before anything runs.

This file runs last (pytest collects it after the other tests) and needs no
state from them, so it also passes alone in a fresh process.
"""
import ctypes

import pytest
import torch

import domain_ring_attention_gb300 as st
from domain_ring_attention_gb300 import _lib
from domain_ring_attention_gb300.workloads import Workload, make_inputs

ST_ERR_SCRATCH_LIMIT = -9


def call_noalloc(lay, q, k, v, causal, out_dtype):
    B, S, H, d = q.shape
    out = torch.empty(q.shape, device=q.device, dtype=out_dtype)
    lse = torch.empty((B, H, S), device=q.device, dtype=torch.float32)
    P = ctypes.c_void_p
    rc = st.load().st_attn_fwd_noalloc(
        lay.handle, B, H, d, _lib._dtype_code(q.dtype), int(causal), 0.0, P(q.data_ptr()),
        P(k.data_ptr()), P(v.data_ptr()), _lib._dtype_code(out_dtype), P(out.data_ptr()),
        P(lse.data_ptr()), P(torch.cuda.current_stream().cuda_stream))
    return rc, out, lse


@pytest.mark.gpu
@pytest.mark.parametrize("d,lens,causal,zigzag", [(128, (1024, 512, 512), True, True),
                                                  (64, (300, 212, 512), False, False)])
def test_noalloc_matches_fwd_on_two_calls(d, lens, causal, zigzag):
    """Two calls in a row on different inputs; the second call's v is a
    thousand times larger, so that a power-of-two scale or a maximum left in
    the shared array by the first call would change the fp16 copy of v and
    hence the output.  Both calls must give, bit for bit, what st_attn_fwd
    gives: the same kernels on the same inputs, only the scratch differs."""
    wl = Workload("noalloc", B=1, H=4, d=d, lens=lens, causal=causal, zigzag=zigzag, dtype="bf16")
    lay = st.Layout(lens, zigzag)
    for seed, v_scale in ((1, 1.0), (2, 1000.0)):
        q, k, v = (x.cuda() for x in make_inputs(wl, seed=seed))
        v = (v.float() * v_scale).to(torch.bfloat16)
        for out_dtype in (torch.bfloat16, torch.float32):
            rc, out, lse = call_noalloc(lay, q, k, v, causal, out_dtype)
            assert rc == 0, _lib.ERRORS.get(rc)
            ref_out, ref_lse = st.st_attn_fwd(lay, q, k, v, causal=causal, out_dtype=out_dtype)
            torch.cuda.synchronize()
            assert st.load().st_device_error(None) == 0
            assert torch.equal(out, ref_out), "out differs from st_attn_fwd (seed %d)" % seed
            assert torch.equal(lse, ref_lse), "lse differs from st_attn_fwd (seed %d)" % seed


def test_noalloc_refuses_problems_beyond_its_scratch():
    """32 MiB holds the fp16 copy of v for B*S*H*d up to ~16.7M elements."""
    lay = st.Layout([8192] * 4)               # S = 32768
    P = ctypes.c_void_p
    good = P(0x10000)
    rc = st.load().st_attn_fwd_noalloc(lay.handle, 1, 8, 128, 1, 1, 0.0, good, good, good, 1, good,
                                       good, None)   # 32768 * 8 * 128 = 33.5M elements
    assert rc == ST_ERR_SCRATCH_LIMIT
    assert "scratch" in st.load().st_error_string(rc).decode()
