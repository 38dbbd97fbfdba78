"""CPU-only checks of the C-ABI library: it loads, exports every symbol the
header declares, builds layouts that agree with the oracle's layout, and
rejects bad arguments with error codes before touching a GPU."""
import ctypes
import os
import re

import numpy as np
import pytest

import domain_ring_attention_gb300 as st
from domain_ring_attention_gb300 import _lib
from oracle import layout as ol

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", f)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names.update(re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(st_\w+)\s*\(", txt, flags=re.M))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_lib.LIB_PATH):
        from domain_ring_attention_gb300 import build
        build.build()
    return st.load()


def test_library_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert "st_attn_fwd" in names and "st_layout_create" in names and len(names) >= 11
    for n in names:
        assert hasattr(lib, n), n
    assert {p[0] for p in _lib.PROTOTYPES} == set(names)


@pytest.mark.parametrize("lens,zigzag", [
    ([100, 150, 130, 132], False), ([16384] * 8, True), ([12928, 19392, 384, 64], True),
    ([2], True), ([1], False), ([7, 1, 3], False), ([2] * 32, True)])
def test_layout_matches_oracle(lib, lens, zigzag):
    lay = st.Layout(lens, zigzag)
    assert lay.S == sum(lens)
    assert lay.offsets() == list(ol.shard_offsets(lens))
    assert np.array_equal(np.array(lay.positions()), ol.natural_positions(lens, zigzag))


@pytest.mark.parametrize("lens,zigzag", [([], False), ([3, 0], False), ([3, 4], True),
                                         ([1] * 33, False), ([-2], False)])
def test_layout_rejects_bad_shapes(lib, lens, zigzag):
    arr = (ctypes.c_int64 * max(1, len(lens)))(*lens)
    h = ctypes.c_void_p()
    rc = lib.st_layout_create(arr, len(lens), int(zigzag), ctypes.byref(h))
    assert rc == -2 and not h.value


def test_layout_null_and_bad_flag(lib):
    h = ctypes.c_void_p()
    assert lib.st_layout_create(None, 1, 0, ctypes.byref(h)) == -1
    arr = (ctypes.c_int64 * 1)(4)
    assert lib.st_layout_create(arr, 1, 2, ctypes.byref(h)) == -8
    assert lib.st_layout_destroy(None) == 0


def test_workspace_sizes(lib):
    lay = st.Layout([100, 150, 130, 132])
    n = ctypes.c_size_t()
    assert lib.st_attn_workspace_size(lay.handle, 1, 2, 64, 0, 0, ctypes.byref(n)) == 0 and n.value == 0
    assert lib.st_attn_workspace_size(lay.handle, 1, 2, 64, 1, 0, ctypes.byref(n)) == 0
    assert n.value >= 512 * 2 * 64 * 2
    assert lib.st_attn_workspace_size(lay.handle, 1, 2, 64, 0, 1, ctypes.byref(n)) == 0
    rows = 512 * 2
    assert n.value >= rows * 64 * 4 + rows * 4
    assert lib.st_attn_workspace_size(lay.handle, 1, 2, 96, 0, 1, ctypes.byref(n)) == -3
    assert lib.st_attn_workspace_size(lay.handle, 1, 2, 64, 7, 1, ctypes.byref(n)) == -3
    assert lib.st_attn_workspace_size(lay.handle, 1, 2, 64, 0, 2, ctypes.byref(n)) == -8


def test_bad_calls_return_codes_without_a_gpu(lib):
    """Validation happens on the host, before any CUDA call."""
    lay = st.Layout([64, 64])
    P = ctypes.c_void_p
    good = P(0x10000)
    lse = P(0x20000)
    fwd = lib.st_attn_fwd
    assert fwd(None, 1, 1, 64, 1, 0, 0.0, good, good, good, 1, good, lse, None, 0, None) == -1
    assert fwd(lay.handle, 1, 1, 64, 1, 0, 0.0, good, good, good, 2, good, lse, good, 1 << 30, None) == -3
    assert fwd(lay.handle, 1, 1, 80, 1, 0, 0.0, good, good, good, 1, good, lse, None, 0, None) == -3
    assert fwd(lay.handle, 1, 1, 64, 5, 0, 0.0, good, good, good, 1, good, lse, None, 0, None) == -3
    assert fwd(lay.handle, 0, 1, 64, 1, 0, 0.0, good, good, good, 1, good, lse, None, 0, None) == -8
    assert fwd(lay.handle, 1, 1, 64, 1, 0, float("nan"), good, good, good, 1, good, lse, None, 0, None) == -8
    assert fwd(lay.handle, 1, 1, 64, 1, 0, 0.0, None, good, good, 1, good, lse, None, 0, None) == -1
    assert fwd(lay.handle, 1, 1, 64, 1, 0, 0.0, P(0x10008), good, good, 1, good, lse, None, 0, None) == -4
    assert fwd(lay.handle, 1, 1, 64, 1, 0, 0.0, good, good, good, 1, good, lse, None, 0, None) == -5
    assert fwd(lay.handle, 1, 1, 64, 1, 0, 0.0, good, good, good, 1, good, lse, good, 64, None) == -5
    bwd = lib.st_attn_bwd
    qkv = [good] * 3
    assert bwd(lay.handle, 1, 1, 64, 1, 0, 0.0, *qkv, good, 1, lse, good, 1, good, good, good, None, 0, None) == -5
    assert bwd(lay.handle, 1, 1, 64, 1, 0, 0.0, *qkv, good, 1, lse, good, 1, good, good, good, good, 16, None) == -5
    assert bwd(lay.handle, 1, 1, 64, 0, 0, 0.0, *qkv, good, 0, lse, good, 1, good, good, good, good, 1 << 30, None) == -3
    assert bwd(lay.handle, 1, 1, 64, 0, 0, 0.0, *qkv, good, 1, lse, good, 0, good, good, good, good, 1 << 30, None) == -3
    fh = lib.st_attn_fwd_host
    h5 = [good] * 5
    d5 = [good, good, good, good, lse]
    assert fh(lay.handle, 1, 1, 64, 1, 0, 0.0, None, good, good, good, lse, *d5, good, 1 << 30, None, good) == -1
    assert fh(lay.handle, 1, 1, 64, 1, 0, 0.0, *h5, good, good, None, good, lse, good, 1 << 30, None, good) == -1
    assert fh(lay.handle, 1, 1, 64, 1, 0, 0.0, *h5, *d5, good, 1 << 30, None, None) == -8    # no copy stream
    assert fh(lay.handle, 1, 1, 64, 1, 0, 0.0, *h5, *d5, good, 1 << 30, good, good) == -8    # the same stream
    assert fh(lay.handle, 1, 1, 64, 0, 0, 0.0, *h5, *d5, good, 1 << 30, None, good) == -3    # fp32
    assert fh(lay.handle, 1, 1, 64, 1, 0, 0.0, *h5, *d5, good, 16, None, good) == -5          # workspace
    assert fh(lay.handle, 1, 1, 64, 1, 0, 0.0, *h5, P(0x10004), *d5[1:], good, 1 << 30, None, good) == -4
    mrg = lib.st_attn_merge
    assert mrg(0, 1, 1, 64, 64, good, good, good, lse, 0, None) == -8
    assert mrg(33, 1, 1, 64, 64, good, good, good, lse, 0, None) == -8
    assert mrg(2, 1, 1, 64, 96, good, good, good, lse, 0, None) == -3
    assert lib.st_permute(lay.handle, 1, 1, 64, 1, 1, good, good, None) == -8
    assert lib.st_error_string(-4).decode().startswith("a tensor pointer")
    gemm = lib.st_proj_gemm
    assert gemm(64, 256, 64, None, good, good, 1, None) == -1
    assert gemm(64, 256, 64, good, good, None, 1, None) == -1
    assert gemm(0, 256, 64, good, good, good, 1, None) == -8
    assert gemm(64, 252, 64, good, good, good, 1, None) == -8      # N not a multiple of 8
    assert gemm(64, 256, 60, good, good, good, 1, None) == -8      # K not a multiple of 8
    assert gemm(64, 256, 64, good, good, good, 2, None) == -3
    assert gemm(64, 256, 64, P(0x10004), good, good, 1, None) == -4
    assert gemm(1 << 30, 1 << 20, 64, good, good, good, 1, None) == -8   # more output tiles than an int counts
    mlp = lib.st_gated_mlp
    w = [good] * 3
    assert mlp(64, 256, 512, None, *w, good, good, 1, None) == -1
    assert mlp(64, 256, 512, good, *w, None, good, 1, None) == -1          # h workspace
    assert mlp(0, 256, 512, good, *w, good, good, 1, None) == -8
    assert mlp(64, 252, 512, good, *w, good, good, 1, None) == -8          # hidden not a multiple of 8
    assert mlp(64, 256, 500, good, *w, good, good, 1, None) == -8          # F not a multiple of 8
    assert mlp(64, 256, 512, good, *w, good, good, 2, None) == -3
    assert mlp(64, 256, 512, good, good, P(0x10004), good, good, good, 1, None) == -4
    rows = (ctypes.c_int64 * 3)(5, 1, 7)
    shards = (P * 3)(0x10000, 0x20000, 0x30000)
    halo = lib.st_halo_exchange
    assert halo(3, None, 16, 64, 1, shards, None) == -1
    assert halo(3, rows, 16, 64, 1, None, None) == -1
    assert halo(0, rows, 16, 64, 1, shards, None) == -8
    assert halo(17, rows, 16, 64, 1, shards, None) == -8            # more shards than ST_CONV_MAX_SHARDS
    assert halo(3, rows, 16, 60, 1, shards, None) == -8             # C not a multiple of 8
    assert halo(3, rows, 16, 64, 4, shards, None) == -8             # halo > 3
    assert halo(3, (ctypes.c_int64 * 3)(5, 0, 7), 16, 64, 1, shards, None) == -2
    assert halo(3, rows, 16, 64, 1, (P * 3)(0x10000, None, 0x30000), None) == -1
    assert halo(3, rows, 16, 64, 1, (P * 3)(0x10000, 0x20008, 0x30000), None) == -4
    conv = lib.st_conv2d_sharded
    outs = (P * 3)(0x40000, 0x50000, 0x60000)
    assert conv(3, rows, 16, 64, 128, 3, shards, None, None, outs, 1, None) == -1
    assert conv(3, rows, 16, 64, 128, 3, shards, good, None, None, 1, None) == -1
    assert conv(3, rows, 16, 64, 128, 4, shards, good, None, outs, 1, None) == -8   # even kernel
    assert conv(3, rows, 16, 64, 128, 9, shards, good, None, outs, 1, None) == -8   # k > 7
    assert conv(3, rows, 16, 96, 128, 3, shards, good, None, outs, 1, None) == -8   # C_in not a multiple of 64
    assert conv(3, rows, 16, 64, 100, 3, shards, good, None, outs, 1, None) == -8   # C_out not a multiple of 8
    assert conv(3, rows, 16, 64, 128, 3, shards, good, None, outs, 2, None) == -3
    assert conv(3, rows, 16, 64, 128, 3, shards, P(0x10004), None, outs, 1, None) == -4
    assert conv(3, rows, 16, 64, 128, 3, shards, good, P(0x10002), outs, 1, None) == -4
    assert conv(3, (ctypes.c_int64 * 3)(1 << 22, 1 << 22, 1 << 22), 1 << 20, 64, 128, 3, shards, good, None, outs,
                1, None) == -8                                              # too many units for an int
    n = ctypes.c_size_t()
    assert lib.st_group_norm_workspace_size(256, 32, ctypes.byref(n)) == 0 and n.value >= 2048 * 32 * 12
    assert lib.st_group_norm_workspace_size(256, 32, None) == -1
    assert lib.st_group_norm_workspace_size(96, 4, ctypes.byref(n)) == -8       # C not a power of two
    assert lib.st_group_norm_workspace_size(256, 64, ctypes.byref(n)) == -8     # 4 channels per group
    gn = lib.st_group_norm_sharded
    ws = P(0x70000)
    big = 1 << 30
    assert gn(3, rows, 16, 256, 32, 1e-5, None, None, None, outs, 0, 1, ws, big, None) == -1
    assert gn(3, rows, 16, 256, 32, 0.0, shards, None, None, outs, 0, 1, ws, big, None) == -8     # eps
    assert gn(3, rows, 16, 256, 32, 1e-5, shards, None, None, outs, 4, 1, ws, big, None) == -8    # out_pad
    assert gn(3, rows, 16, 256, 32, 1e-5, shards, None, None, outs, 0, 2, ws, big, None) == -3
    assert gn(3, rows, 16, 256, 32, 1e-5, shards, None, None, outs, 0, 1, None, big, None) == -5
    assert gn(3, rows, 16, 256, 32, 1e-5, shards, None, None, outs, 0, 1, ws, 64, None) == -5
    assert gn(3, rows, 16, 256, 32, 1e-5, shards, P(0x10002), None, outs, 0, 1, ws, big, None) == -4


def test_python_binding_refuses_cpu_tensors(lib):
    import torch
    lay = st.Layout([4, 4])
    x = torch.zeros(1, 8, 1, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        st.st_attn_fwd(lay, x, x, x)


def test_bindings_refuse_host_memory(lib):
    """Every entry point checks, before it launches, that its device pointers address device memory: host
    tensors come back as ST_ERR_NOT_DEVICE (no GPU is needed to see it)."""
    import types
    import torch
    bf = torch.bfloat16
    x = torch.zeros(64, 64, dtype=bf)
    w = torch.zeros(64, 64, dtype=bf)
    s0 = types.SimpleNamespace(cuda_stream=0)    # the legacy default stream, without asking torch for one
    cases = [
        lambda: st.st_proj_gemm(x, w, stream=s0),
        lambda: st.st_gated_mlp(x, w, w, w, stream=s0),
        lambda: st.st_halo_exchange([torch.zeros(6, 8, 64, dtype=bf), torch.zeros(5, 8, 64, dtype=bf)], 1, stream=s0),
        lambda: st.st_conv2d_sharded([torch.zeros(6, 8, 64, dtype=bf)], torch.zeros(64, 3, 3, 64, dtype=bf),
                                     stream=s0),
        lambda: st.st_group_norm_sharded([torch.zeros(4, 8, 64, dtype=bf)], 8, stream=s0),
    ]
    for call in cases:
        with pytest.raises(st.StAttnError) as e:
            call()
        assert e.value.code == -10, e.value
    assert lib.st_is_device_pointer(ctypes.c_void_p(x.data_ptr())) == 0
    assert lib.st_error_string(-10).decode().startswith("a pointer that must address device memory")


def test_bounded_wait_selftest_rejects_bad_limits(lib):
    """The wait limit is checked on the host before anything is launched."""
    assert lib.st_selftest_bounded_wait(0, None) == -8
    assert lib.st_selftest_bounded_wait(-5, None) == -8
    assert lib.st_selftest_bounded_wait(5 * 10 ** 9, None) == -8


def test_ring_entry_points_check_arguments_on_the_host(lib):
    lay = st.Layout([256, 128, 384], True)
    n = ctypes.c_size_t()
    for which in range(4):
        assert lib.st_ring_workspace_size(lay.handle, 1, 2, 128, which, ctypes.byref(n)) == 0 and n.value > 0
    assert lib.st_ring_workspace_size(lay.handle, 1, 2, 128, 4, ctypes.byref(n)) == -8
    assert lib.st_ring_workspace_size(lay.handle, 1, 2, 96, 0, ctypes.byref(n)) == -3
    P = ctypes.c_void_p
    good = P(0x10000)
    args = lambda qs, ks, dt: (lay.handle, qs, ks, 1, 2, 128, dt, 1, 0.0, good, good, good, None, None, 0, good,
                               good, good, 1 << 30, None)
    assert lib.st_ring_fwd_step(*args(3, 0, 1)) == -8          # shard index out of range
    assert lib.st_ring_fwd_step(*args(0, -1, 1)) == -8
    assert lib.st_ring_fwd_step(*args(0, 1, 0)) == -3          # fp32: not a ring-step dtype
    a = list(args(0, 1, 1))
    a[12] = good                                               # prev_out without prev_lse
    assert lib.st_ring_fwd_step(*a) == -1
    a = list(args(0, 1, 1))
    a[18] = 16                                                 # workspace too small
    assert lib.st_ring_fwd_step(*a) == -5
    arr = (P * 3)(good, good, good)
    # copy stream missing
    assert lib.st_ring_fwd_local(lay.handle, 1, 2, 128, 1, 0.0, arr, arr, arr, 1, arr, arr, good, 1 << 40,
                                 None, None) == -8
