"""The device-pointer check every entry point applies before it launches (st_is_device_pointer).

Only the check itself is called here: no kernel is ever launched with a host pointer.
"""
import ctypes

import numpy as np
import pytest
import torch

import domain_ring_attention_gb300 as st

pytestmark = pytest.mark.gpu


def test_device_pointer_check():
    lib = st.load()
    dev = torch.empty(1024, device="cuda")
    pinned = torch.empty(1024, pin_memory=True)
    pageable = np.zeros(1024, dtype=np.float32)
    assert lib.st_is_device_pointer(ctypes.c_void_p(dev.data_ptr())) == 1
    assert lib.st_is_device_pointer(ctypes.c_void_p(dev.data_ptr() + 256)) == 1
    assert lib.st_is_device_pointer(ctypes.c_void_p(pinned.data_ptr())) == 0
    assert lib.st_is_device_pointer(ctypes.c_void_p(pageable.ctypes.data)) == 0
    assert lib.st_is_device_pointer(None) == 0
    # the failed queries leave no CUDA error behind for a later launch check to pick up
    assert torch.cuda.is_available()
    x = torch.ones(8, device="cuda")
    torch.cuda.synchronize()
    assert float(x.sum()) == 8.0
