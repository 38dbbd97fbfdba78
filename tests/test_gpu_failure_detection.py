"""Failure detection on the GPU without a fault: a bounded device wait that runs out.

Every barrier wait of the tensor-core kernels gives up after a bounded number of clock cycles, records the timeout
in a device error word and lets the kernel return; st_device_error reports it to the host.  Here a one-CTA kernel
waits, with a short limit, on an mbarrier that nothing arrives at, with no copy, MMA or tensor memory in flight.
The timeout must be reported once, cleared by the report, and the context must stay usable.
"""
import ctypes

import pytest
import torch

import domain_ring_attention_gb300 as st
from domain_ring_attention_gb300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu

ST_ERR_DEVICE_TIMEOUT = -7


def test_bounded_wait_runs_out_and_is_reported():
    lib = st.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.st_device_error(stream) == 0            # nothing pending from earlier work
    assert lib.st_selftest_bounded_wait(100000, stream) == 0   # ~50 us of polling at 2 GHz
    assert lib.st_device_error(stream) == ST_ERR_DEVICE_TIMEOUT
    assert lib.st_device_error(stream) == 0            # the report cleared the word
    # the context still runs the attention kernels, and they report no timeout
    wl = Workload("after", B=1, H=2, d=64, lens=(256, 256), causal=True, zigzag=True, dtype="bf16")
    q, k, v = (x.cuda() for x in make_inputs(wl, seed=1))
    lay = st.Layout(wl.lens, True)
    o1, l1 = st.st_attn_fwd(lay, q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.isfinite(o1.float()).all() and torch.isfinite(l1).all()
    assert lib.st_device_error(stream) == 0

