"""ctypes binding of the C-ABI in include/st_attn.h.

Argument marshalling only: every step of the computation runs inside the
CUDA library.  PyTorch provides device memory and the current stream.  If the
library has not been built, loading fails with an error; there is no other
implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# ST_ATTN_LIB may name another build of the same library (e.g. one made with
# other compiler flags); by default the in-tree build is loaded.
LIB_PATH = os.environ.get("ST_ATTN_LIB") or os.path.join(_PKG, "lib", "libst_attn.so")

ST_DTYPE_F32 = 0
ST_DTYPE_BF16 = 1
ST_MAX_SHARDS = 32
ST_CONV_MAX_SHARDS = 16

ERRORS = {
    0: "ST_OK", -1: "ST_ERR_NULL", -2: "ST_ERR_INVALID_LAYOUT", -3: "ST_ERR_UNSUPPORTED",
    -4: "ST_ERR_MISALIGNED", -5: "ST_ERR_WORKSPACE", -6: "ST_ERR_CUDA",
    -7: "ST_ERR_DEVICE_TIMEOUT", -8: "ST_ERR_INVALID_ARG", -9: "ST_ERR_SCRATCH_LIMIT",
    -10: "ST_ERR_NOT_DEVICE",
}

# C prototypes: (name, restype, argtypes)
_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_F = ctypes.c_float
_SZ = ctypes.c_size_t
PROTOTYPES = [
    ("st_layout_create", _I, [ctypes.POINTER(_I64), _I, _I, ctypes.POINTER(_P)]),
    ("st_layout_destroy", _I, [_P]),
    ("st_layout_query", _I, [_P, ctypes.POINTER(_I64), ctypes.POINTER(_I64), ctypes.POINTER(_I64),
                             ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    ("st_attn_workspace_size", _I, [_P, _I, _I, _I, _I, _I, ctypes.POINTER(_SZ)]),
    ("st_attn_fwd", _I, [_P, _I, _I, _I, _I, _I, _F, _P, _P, _P, _I, _P, _P, _P, _SZ, _P]),
    ("st_attn_fwd_host", _I, [_P, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                              _P, _P]),
    ("st_attn_fwd_noalloc", _I, [_P, _I, _I, _I, _I, _I, _F, _P, _P, _P, _I, _P, _P, _P]),
    ("st_attn_fwd_partials", _I, [_P, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    ("st_attn_merge", _I, [_I, _I, _I, _I64, _I, _P, _P, _P, _P, _I, _P]),
    ("st_attn_bwd", _I, [_P, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _I, _P, _P, _I, _P, _P, _P,
                         _P, _SZ, _P]),
    ("st_permute", _I, [_P, _I, _I, _I, _I, _I, _P, _P, _P]),
    ("st_proj_gemm", _I, [_I, _I, _I, _P, _P, _P, _I, _P]),
    ("st_is_device_pointer", _I, [_P]),
    ("st_gated_mlp", _I, [_I, _I, _I, _P, _P, _P, _P, _P, _P, _I, _P]),
    ("st_halo_exchange", _I, [_I, ctypes.POINTER(_I64), _I, _I, _I, ctypes.POINTER(_P), _P]),
    ("st_conv2d_sharded", _I, [_I, ctypes.POINTER(_I64), _I, _I, _I, _I, ctypes.POINTER(_P), _P, _P,
                               ctypes.POINTER(_P), _I, _P]),
    ("st_group_norm_workspace_size", _I, [_I, _I, ctypes.POINTER(_SZ)]),
    ("st_group_norm_sharded", _I, [_I, ctypes.POINTER(_I64), _I, _I, _I, _F, ctypes.POINTER(_P), _P, _P,
                                   ctypes.POINTER(_P), _I, _I, _P, _SZ, _P]),
    ("st_error_string", ctypes.c_char_p, [_I]),
    ("st_last_cuda_error", _I, []),
    ("st_device_error", _I, [_P]),
    ("st_selftest_bounded_wait", _I, [ctypes.c_longlong, _P]),
    ("st_ring_workspace_size", _I, [_P, _I, _I, _I, _I, ctypes.POINTER(_SZ)]),
    ("st_attn_bwd_delta", _I, [_I, _I, _I64, _I, _I, _P, _I, _P, _P, _P]),
    ("st_convert_f32", _I, [_I64, _P, _P, _I, _P]),
    ("st_fp16_scaled_copy", _I, [_I64, _P, _P, _P, _P, _P]),
    ("st_ring_fwd_step", _I, [_P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P, _I, _P, _P, _P, _SZ, _P]),
    ("st_ring_bwd_step", _I, [_P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _I, _P, _P, _I, _P, _P, _P,
                              _P, _SZ, _P]),
    ("st_ring_fwd_local", _I, [_P, _I, _I, _I, _I, _F, ctypes.POINTER(_P), ctypes.POINTER(_P), ctypes.POINTER(_P),
                               _I, ctypes.POINTER(_P), ctypes.POINTER(_P), _P, _SZ, _P, _P]),
    ("st_ring_bwd_local", _I, [_P, _I, _I, _I, _I, _F, ctypes.POINTER(_P), ctypes.POINTER(_P), ctypes.POINTER(_P),
                               ctypes.POINTER(_P), _I, ctypes.POINTER(_P), ctypes.POINTER(_P), ctypes.POINTER(_P),
                               ctypes.POINTER(_P), ctypes.POINTER(_P), _P, _SZ, _P, _P]),
]

_lib = None


class StAttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = "%s failed: %s (%d)" % (where, ERRORS.get(code, "?"), code)
        if _lib is not None:
            msg += ": " + _lib.st_error_string(code).decode()
            if code == -6:
                msg += " [cudaError %d]" % _lib.st_last_cuda_error()
        super().__init__(msg)


def load():
    """Load the shared library (once).  Raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libst_attn.so is not built (run __graft_entry__.build() "
                               "or python -m domain_ring_attention_gb300.build)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, res, args in PROTOTYPES:
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(rc: int, where: str):
    if rc != 0:
        raise StAttnError(rc, where)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(stream, *keep):
    """The handle of the stream a call runs on.  ``keep``: device tensors the call's kernels use that this
    binding allocated (workspaces, outputs).  The caching allocator ties a block to the stream that was current
    at its allocation; when the call runs on another stream they are recorded on it, so that their memory is
    not handed to other work before the call's kernels are done with it."""
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    held = [x for t in keep for x in (t if isinstance(t, (list, tuple)) else (t,)) if x is not None and x.is_cuda]
    if held and stream != torch.cuda.current_stream(held[0].device):
        for x in held:
            x.record_stream(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(dt):
    if dt == torch.float32:
        return ST_DTYPE_F32
    if dt == torch.bfloat16:
        return ST_DTYPE_BF16
    raise TypeError("only float32 and bfloat16 tensors are supported, got %s" % dt)


class Layout:
    """Owner of an ``st_layout_t`` built from sharding shapes."""

    def __init__(self, shard_lens, zigzag: bool = False):
        lib = load()
        lens = [int(x) for x in shard_lens]
        arr = (_I64 * max(1, len(lens)))(*lens)
        h = ctypes.c_void_p()
        _check(lib.st_layout_create(arr, len(lens), int(bool(zigzag)), ctypes.byref(h)),
               "st_layout_create")
        self._h = h
        self.lens = lens
        self.zigzag = bool(zigzag)
        S = _I64()
        _check(lib.st_layout_query(h, ctypes.byref(S), None, None, None, None), "st_layout_query")
        self.S = int(S.value)
        self.D = len(lens)

    @property
    def handle(self):
        return self._h

    def offsets(self):
        lib = load()
        off = (_I64 * (self.D + 1))()
        _check(lib.st_layout_query(self._h, None, off, None, None, None), "st_layout_query")
        return [int(x) for x in off]

    def positions(self):
        lib = load()
        pos = (_I64 * self.S)()
        _check(lib.st_layout_query(self._h, None, None, pos, None, None), "st_layout_query")
        return list(pos)

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            load().st_layout_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _shape(q):
    if q.dim() != 4:
        raise ValueError("expected a [B, S, H, d] tensor")
    return tuple(int(x) for x in q.shape)


def _check_tensor(t, shape, dtype, name):
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype or not t.is_contiguous():
        raise ValueError("%s must be contiguous %s of shape %s" % (name, dtype, tuple(shape)))


def st_attn_workspace_size(layout, B, H, d, dtype, pass_):
    n = _SZ()
    _check(load().st_attn_workspace_size(layout.handle, B, H, d, _dtype_code(dtype), pass_,
                                         ctypes.byref(n)), "st_attn_workspace_size")
    return int(n.value)


def st_attn_fwd(layout, q, k, v, causal=False, scale=0.0, out=None, lse=None, stream=None,
                out_dtype=None, workspace=None):
    """out, lse = attention of buffer-order BSHD q, k, v under ``layout``.

    ``out_dtype`` defaults to the input dtype; torch.float32 returns the
    normalised fp32 accumulator without the final rounding.  ``workspace``
    (uint8 device tensor of ``st_attn_workspace_size(..., 0)`` bytes) is
    allocated here when not given.
    """
    B, S, H, d = _shape(q)
    for t, n in ((k, "k"), (v, "v")):
        _check_tensor(t, q.shape, q.dtype, n)
    _check_tensor(q, q.shape, q.dtype, "q")
    odt = (out.dtype if out is not None else q.dtype) if out_dtype is None else out_dtype
    if out is None:
        out = torch.empty(q.shape, device=q.device, dtype=odt)
    if lse is None:
        lse = torch.empty((B, H, S), device=q.device, dtype=torch.float32)
    _check_tensor(out, q.shape, odt, "out")
    _check_tensor(lse, (B, H, S), torch.float32, "lse")
    if workspace is None:
        need = st_attn_workspace_size(layout, B, H, d, q.dtype, 0)
        workspace = torch.empty(max(need, 1), device=q.device, dtype=torch.uint8)
    _check(load().st_attn_fwd(layout.handle, B, H, d, _dtype_code(q.dtype), int(bool(causal)),
                              float(scale), _ptr(q), _ptr(k), _ptr(v), _dtype_code(odt), _ptr(out),
                              _ptr(lse), _ptr(workspace), workspace.numel(), _stream(stream, out, lse, workspace)),
           "st_attn_fwd")
    return out, lse


def st_attn_fwd_host(layout, q_host, k_host, v_host, out_host, lse_host, dev, causal=False, scale=0.0,
                     workspace=None, stream=None, copy_stream=None):
    """st_attn_fwd from host buffers with the copies overlapped with compute
    (bf16 only).  ``q_host``, ``k_host``, ``v_host``, ``out_host`` are CPU
    [B,S,H,d] bf16 tensors (pinned for overlap), ``lse_host`` CPU [B,H,S]
    fp32; ``dev`` is a dict of device staging tensors ``q``, ``k``, ``v``,
    ``out`` (same shape) and ``lse``.  ``copy_stream`` (a torch.cuda.Stream
    other than ``stream``) carries the copies; it is created when not given.
    When ``stream`` completes, out_host and lse_host hold the results."""
    B, S, H, d = _shape(q_host)
    for t, n in ((q_host, "q_host"), (k_host, "k_host"), (v_host, "v_host"), (out_host, "out_host")):
        if t.is_cuda or tuple(t.shape) != (B, S, H, d) or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CPU bf16 tensor of shape %s" % (n, (B, S, H, d)))
    if lse_host.is_cuda or tuple(lse_host.shape) != (B, H, S) or lse_host.dtype != torch.float32 \
            or not lse_host.is_contiguous():
        raise ValueError("lse_host must be a contiguous CPU fp32 tensor of shape %s" % ((B, H, S),))
    for n in ("q", "k", "v", "out"):
        _check_tensor(dev[n], (B, S, H, d), torch.bfloat16, n)
    _check_tensor(dev["lse"], (B, H, S), torch.float32, "lse")
    if workspace is None:
        need = st_attn_workspace_size(layout, B, H, d, torch.bfloat16, 0)
        workspace = torch.empty(max(need, 1), device=dev["q"].device, dtype=torch.uint8)
    if stream is None:
        stream = torch.cuda.current_stream()
    if copy_stream is None:
        copy_stream = torch.cuda.Stream(device=dev["q"].device)
    _check(load().st_attn_fwd_host(layout.handle, B, H, d, ST_DTYPE_BF16, int(bool(causal)), float(scale),
                                   _ptr(q_host), _ptr(k_host), _ptr(v_host), _ptr(out_host), _ptr(lse_host),
                                   _ptr(dev["q"]), _ptr(dev["k"]), _ptr(dev["v"]), _ptr(dev["out"]),
                                   _ptr(dev["lse"]), _ptr(workspace), workspace.numel(),
                                   _stream(stream, workspace), _stream(copy_stream)), "st_attn_fwd_host")
    return out_host, lse_host


def st_attn_fwd_partials(layout, q, k, v, causal=False, scale=0.0, stream=None, workspace=None):
    """Per-KV-shard partials: (partial_out [D,B,S,H,d] fp32, partial_lse [D,B,H,S]).
    ``workspace`` as st_attn_fwd (allocated here when not given)."""
    B, S, H, d = _shape(q)
    D = layout.D
    po = torch.empty((D, B, S, H, d), device=q.device, dtype=torch.float32)
    pl = torch.empty((D, B, H, S), device=q.device, dtype=torch.float32)
    if workspace is None:
        need = st_attn_workspace_size(layout, B, H, d, q.dtype, 0)
        workspace = torch.empty(max(need, 1), device=q.device, dtype=torch.uint8)
    _check(load().st_attn_fwd_partials(layout.handle, B, H, d, _dtype_code(q.dtype),
                                       int(bool(causal)), float(scale), _ptr(q), _ptr(k), _ptr(v),
                                       _ptr(po), _ptr(pl), _ptr(workspace), workspace.numel(),
                                       _stream(stream, po, pl, workspace)), "st_attn_fwd_partials")
    return po, pl


def st_attn_merge(partial_out, partial_lse, out_dtype=torch.float32, out=None, lse=None,
                  stream=None):
    """Log-sum-exp merge of D partials -> (out [B,S,H,d], lse [B,H,S])."""
    D, B, S, H, d = (int(x) for x in partial_out.shape)
    _check_tensor(partial_out, (D, B, S, H, d), torch.float32, "partial_out")
    _check_tensor(partial_lse, (D, B, H, S), torch.float32, "partial_lse")
    if out is None:
        out = torch.empty((B, S, H, d), device=partial_out.device, dtype=out_dtype)
    if lse is None:
        lse = torch.empty((B, H, S), device=partial_out.device, dtype=torch.float32)
    _check(load().st_attn_merge(D, B, H, S, d, _ptr(partial_out), _ptr(partial_lse), _ptr(out),
                                _ptr(lse), _dtype_code(out.dtype), _stream(stream, out, lse)), "st_attn_merge")
    return out, lse


def st_attn_bwd(layout, q, k, v, out, lse, dout, causal=False, scale=0.0, grad_dtype=None,
                workspace=None, stream=None):
    """dq, dk, dv of sum(dout * out), in ``grad_dtype`` (default: fp32).

    ``out`` is the forward output in the input dtype or in fp32.
    """
    B, S, H, d = _shape(q)
    for t, n in ((k, "k"), (v, "v"), (dout, "dout")):
        _check_tensor(t, q.shape, q.dtype, n)
    if out.dtype != torch.float32:
        _check_tensor(out, q.shape, q.dtype, "out")
    else:
        _check_tensor(out, q.shape, torch.float32, "out")
    _check_tensor(lse, (B, H, S), torch.float32, "lse")
    need = st_attn_workspace_size(layout, B, H, d, q.dtype, 1)
    if workspace is None:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    gdt = torch.float32 if grad_dtype is None else grad_dtype
    dq, dk, dv = (torch.empty(q.shape, device=q.device, dtype=gdt) for _ in range(3))
    _check(load().st_attn_bwd(layout.handle, B, H, d, _dtype_code(q.dtype), int(bool(causal)),
                              float(scale), _ptr(q), _ptr(k), _ptr(v), _ptr(out),
                              _dtype_code(out.dtype), _ptr(lse), _ptr(dout), _dtype_code(gdt),
                              _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                              workspace.numel() * workspace.element_size(),
                              _stream(stream, dq, dk, dv, workspace)),
           "st_attn_bwd")
    return dq, dk, dv


def st_permute(layout, x, to_natural=True, stream=None):
    B, S, H, d = _shape(x)
    out = torch.empty_like(x)
    _check(load().st_permute(layout.handle, B, H, d, _dtype_code(x.dtype), int(bool(to_natural)),
                             _ptr(x), _ptr(out), _stream(stream, out)), "st_permute")
    return out


def st_proj_gemm(x, w, out_dtype=torch.bfloat16, out=None, stream=None):
    """Projection y = x w^T on the tensor cores: x [M, K] bf16, w [N, K] bf16
    (a Linear layer's [out, in] weight) -> y [M, N] in ``out_dtype``.  Leading
    dimensions of x are flattened (x [..., K] gives y [..., N])."""
    if x.dtype != torch.bfloat16 or w.dtype != torch.bfloat16:
        raise StAttnError(-3, "st_proj_gemm (bf16 inputs)")
    if not x.is_contiguous() or not w.is_contiguous():
        raise StAttnError(-8, "st_proj_gemm (contiguous inputs)")
    K = int(x.shape[-1])
    M = x.numel() // max(K, 1)
    N = int(w.shape[0])
    if w.dim() != 2 or int(w.shape[1]) != K:
        raise StAttnError(-8, "st_proj_gemm (weight shape)")
    if out is None:
        out = torch.empty(tuple(x.shape[:-1]) + (N,), device=x.device, dtype=out_dtype)
    _check(load().st_proj_gemm(M, N, K, _ptr(x), _ptr(w), _ptr(out), _dtype_code(out.dtype),
                               _stream(stream, out)),
           "st_proj_gemm")
    return out


def st_gated_mlp(x, w1, w3, w2, out_dtype=torch.bfloat16, out=None, h=None, stream=None):
    """Gated MLP y = (silu(x w1^T) * (x w3^T)) w2^T on the tensor cores:
    x [..., hidden] bf16, w1 and w3 [F, hidden] bf16, w2 [hidden, F] bf16 ->
    y [..., hidden] in ``out_dtype``.  ``h`` ([M, F] bf16) receives the gated
    activation; it is allocated when not given.  Returns (y, h)."""
    ws = (x, w1, w3, w2)
    if any(t.dtype != torch.bfloat16 for t in ws):
        raise StAttnError(-3, "st_gated_mlp (bf16 inputs)")
    if not all(t.is_contiguous() for t in ws):
        raise StAttnError(-8, "st_gated_mlp (contiguous inputs)")
    hidden = int(x.shape[-1])
    M = x.numel() // max(hidden, 1)
    F = int(w1.shape[0])
    if (w1.dim() != 2 or tuple(w1.shape) != (F, hidden) or tuple(w3.shape) != (F, hidden)
            or tuple(w2.shape) != (hidden, F)):
        raise StAttnError(-8, "st_gated_mlp (weight shapes)")
    if h is None:
        h = torch.empty((M, F), device=x.device, dtype=torch.bfloat16)
    elif h.dtype != torch.bfloat16 or h.numel() != M * F or not h.is_contiguous():
        raise StAttnError(-8, "st_gated_mlp (h workspace)")
    if out is None:
        out = torch.empty(tuple(x.shape[:-1]) + (hidden,), device=x.device, dtype=out_dtype)
    _check(load().st_gated_mlp(M, hidden, F, _ptr(x), _ptr(w1), _ptr(w3), _ptr(w2), _ptr(h), _ptr(out),
                               _dtype_code(out.dtype), _stream(stream, out, h)), "st_gated_mlp")
    return out, h


def _ptr_array(ts):
    return (_P * len(ts))(*[t.data_ptr() for t in ts])


def _image_shards(shards, pad, name):
    """Shard lengths and the common (W, C) of a list of channels-last shards
    [L_r + 2*pad, W, C]."""
    if not shards:
        raise StAttnError(-8, name + " (no shards)")
    W, C = int(shards[0].shape[1]), int(shards[0].shape[2])
    rows = []
    for t in shards:
        if t.dim() != 3 or int(t.shape[1]) != W or int(t.shape[2]) != C or not t.is_contiguous():
            raise StAttnError(-8, name + " (shards must be contiguous [rows, W, C] with one W and C)")
        rows.append(int(t.shape[0]) - 2 * pad)
    return rows, W, C


def st_halo_exchange(shards, halo, stream=None):
    """Fill, in place, the ``halo`` pad rows above and below every shard of a
    row-sharded image.  ``shards``: list of D bf16 tensors [L_r + 2*halo, W, C]
    (channels last) whose middle L_r rows hold the shard's image rows, in
    order.  Pad rows receive the neighbouring image rows (zeros outside the
    image).  Returns ``shards``."""
    if any(t.dtype != torch.bfloat16 for t in shards):
        raise StAttnError(-3, "st_halo_exchange (bf16 shards)")
    rows, W, C = _image_shards(shards, halo, "st_halo_exchange")
    D = len(shards)
    _check(load().st_halo_exchange(D, (_I64 * D)(*rows), W, C, int(halo), _ptr_array(shards), _stream(stream)),
           "st_halo_exchange")
    return shards


def st_conv2d_sharded(shards, weight, bias=None, out_dtype=torch.bfloat16, out=None, stream=None):
    """2-D convolution (cross-correlation, stride 1, zero padding (k-1)/2) of a
    row-sharded image from halo-padded shards, one output per shard.
    ``shards``: list of D bf16 tensors [L_r + k - 1, W, C_in] after
    st_halo_exchange(shards, (k-1)//2); ``weight``: bf16 [C_out, k, k, C_in];
    ``bias``: fp32 [C_out] or None.  Returns the list of [L_r, W, C_out]."""
    if weight.dtype != torch.bfloat16 or any(t.dtype != torch.bfloat16 for t in shards):
        raise StAttnError(-3, "st_conv2d_sharded (bf16 inputs)")
    if weight.dim() != 4 or weight.shape[1] != weight.shape[2] or not weight.is_contiguous():
        raise StAttnError(-8, "st_conv2d_sharded (weight [C_out, k, k, C_in])")
    C_out, k, C_in = int(weight.shape[0]), int(weight.shape[1]), int(weight.shape[3])
    rows, W, C = _image_shards(shards, (k - 1) // 2, "st_conv2d_sharded")
    if C != C_in:
        raise StAttnError(-8, "st_conv2d_sharded (channels of shards and weight differ)")
    if bias is not None and (bias.dtype != torch.float32 or bias.numel() != C_out or not bias.is_contiguous()):
        raise StAttnError(-8, "st_conv2d_sharded (bias fp32 [C_out])")
    if out is None:
        out = [torch.empty((max(L, 0), W, C_out), device=shards[0].device, dtype=out_dtype) for L in rows]
    D = len(shards)
    _check(load().st_conv2d_sharded(D, (_I64 * D)(*rows), W, C_in, C_out, k, _ptr_array(shards), _ptr(weight),
                                    _ptr(bias), _ptr_array(out), _dtype_code(out[0].dtype), _stream(stream, out)),
           "st_conv2d_sharded")
    return out


def st_group_norm_sharded(shards, G, gamma=None, beta=None, eps=1e-5, out_dtype=torch.bfloat16, out=None,
                          out_pad=0, workspace=None, stream=None):
    """Group normalisation of a row-sharded image with statistics combined
    over all shards.  ``shards``: list of D bf16 tensors [L_r, W, C];
    ``gamma``/``beta``: fp32 [C] or None.  Returns the list of outputs
    [L_r + 2*out_pad, W, C] (pad rows untouched)."""
    if any(t.dtype != torch.bfloat16 for t in shards):
        raise StAttnError(-3, "st_group_norm_sharded (bf16 shards)")
    rows, W, C = _image_shards(shards, 0, "st_group_norm_sharded")
    for name, t in (("gamma", gamma), ("beta", beta)):
        if t is not None and (t.dtype != torch.float32 or t.numel() != C or not t.is_contiguous()):
            raise StAttnError(-8, "st_group_norm_sharded (%s fp32 [C])" % name)
    lib = load()
    n = ctypes.c_size_t()
    _check(lib.st_group_norm_workspace_size(C, int(G), ctypes.byref(n)), "st_group_norm_workspace_size")
    if workspace is None:
        workspace = torch.empty(n.value, device=shards[0].device, dtype=torch.uint8)
    if out is None:
        out = [torch.zeros((L + 2 * out_pad, W, C), device=shards[0].device, dtype=out_dtype) for L in rows]
    D = len(shards)
    _check(lib.st_group_norm_sharded(D, (_I64 * D)(*rows), W, C, int(G), float(eps), _ptr_array(shards),
                                     _ptr(gamma), _ptr(beta), _ptr_array(out), int(out_pad),
                                     _dtype_code(out[0].dtype), _ptr(workspace), workspace.numel(),
                                     _stream(stream, out, workspace)), "st_group_norm_sharded")
    return out


# ---------------------------------------------------------------- ring attention across ranks

def st_ring_workspace_size(layout, B, H, d, which):
    n = _SZ()
    _check(load().st_ring_workspace_size(layout.handle, B, H, d, which, ctypes.byref(n)),
           "st_ring_workspace_size")
    return int(n.value)


def st_ring_fwd_step(layout, q_shard, kv_shard, q, k, v, prev=None, causal=False, scale=0.0,
                     out_dtype=torch.float32, out=None, lse=None, workspace=None, stream=None):
    """One ring step of rank ``q_shard``: q [B, L_q, H, d] against the K/V block
    [B, L_kv, H, d] of shard ``kv_shard`` (bf16), merged into ``prev`` (a pair
    (out fp32, lse) of the running state, or None at the first step).
    Returns (out, lse); out may be ``prev[0]`` itself (fp32)."""
    B, Lq, H, d = _shape(q)
    Lkv = int(k.shape[1])
    _check_tensor(q, (B, Lq, H, d), torch.bfloat16, "q")
    _check_tensor(k, (B, Lkv, H, d), torch.bfloat16, "k")
    _check_tensor(v, (B, Lkv, H, d), torch.bfloat16, "v")
    if out is None:
        out = torch.empty((B, Lq, H, d), device=q.device, dtype=out_dtype)
    if lse is None:
        lse = torch.empty((B, H, Lq), device=q.device, dtype=torch.float32)
    if workspace is None:
        workspace = torch.empty(st_ring_workspace_size(layout, B, H, d, 0), device=q.device, dtype=torch.uint8)
    po, pl = (None, None) if prev is None else prev
    _check(load().st_ring_fwd_step(layout.handle, int(q_shard), int(kv_shard), B, H, d, ST_DTYPE_BF16,
                                   int(bool(causal)), float(scale), _ptr(q), _ptr(k), _ptr(v), _ptr(po), _ptr(pl),
                                   _dtype_code(out.dtype), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
                                   _stream(stream, out, lse, workspace)), "st_ring_fwd_step")
    return out, lse


def st_ring_bwd_step(layout, q_shard, kv_shard, q, k, v, out, lse, dout, dq, dk, dv, first_q, causal=False,
                     scale=0.0, workspace=None, stream=None):
    """One backward ring step: adds the block's contributions to the fp32
    ``dq`` (zeroed first when ``first_q``), ``dk`` and ``dv``."""
    B, Lq, H, d = _shape(q)
    if workspace is None:
        workspace = torch.empty(st_ring_workspace_size(layout, B, H, d, 1), device=q.device, dtype=torch.uint8)
    _check(load().st_ring_bwd_step(layout.handle, int(q_shard), int(kv_shard), B, H, d, ST_DTYPE_BF16,
                                   int(bool(causal)), float(scale), _ptr(q), _ptr(k), _ptr(v), _ptr(out),
                                   _dtype_code(out.dtype), _ptr(lse), _ptr(dout), int(bool(first_q)), _ptr(dq),
                                   _ptr(dk), _ptr(dv), _ptr(workspace), workspace.numel(), _stream(stream, workspace)),
           "st_ring_bwd_step")
    return dq, dk, dv


def _ptrs(ts):
    return (_P * len(ts))(*[t.data_ptr() for t in ts])


def st_ring_fwd_local(layout, qs, ks, vs, causal=False, scale=0.0, out_dtype=torch.bfloat16, stream=None,
                      copy_stream=None, workspace=None):
    """The ring forward with the D ranks on this GPU: lists of per-rank shards
    qs, ks, vs ([B, L_r, H, d] bf16).  Returns (outs, lses), per rank."""
    D = layout.D
    B, _, H, d = _shape(qs[0])
    dev = qs[0].device
    outs = [torch.empty((B, L, H, d), device=dev, dtype=out_dtype) for L in layout.lens]
    lses = [torch.empty((B, H, L), device=dev, dtype=torch.float32) for L in layout.lens]
    if workspace is None:
        workspace = torch.empty(st_ring_workspace_size(layout, B, H, d, 2), device=dev, dtype=torch.uint8)
    if copy_stream is None:
        copy_stream = torch.cuda.Stream(device=dev)
    _check(load().st_ring_fwd_local(layout.handle, B, H, d, int(bool(causal)), float(scale), _ptrs(qs), _ptrs(ks),
                                    _ptrs(vs), _dtype_code(out_dtype), _ptrs(outs), _ptrs(lses), _ptr(workspace),
                                    workspace.numel(), _stream(stream, outs, lses, workspace), _stream(copy_stream)),
           "st_ring_fwd_local")
    return outs, lses


def st_ring_bwd_local(layout, qs, ks, vs, outs, lses, douts, causal=False, scale=0.0, stream=None,
                      copy_stream=None, workspace=None):
    """The ring backward with the D ranks on this GPU.  Returns per-rank fp32
    (dqs, dks, dvs)."""
    B, _, H, d = _shape(qs[0])
    dev = qs[0].device
    mk = lambda: [torch.empty((B, L, H, d), device=dev, dtype=torch.float32) for L in layout.lens]
    dqs, dks, dvs = mk(), mk(), mk()
    if workspace is None:
        workspace = torch.empty(st_ring_workspace_size(layout, B, H, d, 3), device=dev, dtype=torch.uint8)
    if copy_stream is None:
        copy_stream = torch.cuda.Stream(device=dev)
    _check(load().st_ring_bwd_local(layout.handle, B, H, d, int(bool(causal)), float(scale), _ptrs(qs), _ptrs(ks),
                                    _ptrs(vs), _ptrs(outs), _dtype_code(outs[0].dtype), _ptrs(lses), _ptrs(douts),
                                    _ptrs(dqs), _ptrs(dks), _ptrs(dvs), _ptr(workspace), workspace.numel(),
                                    _stream(stream, dqs, dks, dvs, workspace), _stream(copy_stream)), "st_ring_bwd_local")
    return dqs, dks, dvs


# ---------------------------------------------------------------- the backward's HBM-bound steps on their own

def st_attn_bwd_delta(out, dout, delta=None, stream=None):
    """Delta [B, H, S] fp32 = rowsum(dout * out) of BSHD tensors (out bf16 or fp32, dout bf16 or fp32)."""
    B, S, H, d = _shape(dout)
    if delta is None:
        delta = torch.empty((B, H, S), device=dout.device, dtype=torch.float32)
    _check(load().st_attn_bwd_delta(B, H, S, d, _dtype_code(dout.dtype), _ptr(out), _dtype_code(out.dtype),
                                    _ptr(dout), _ptr(delta), _stream(stream, delta)), "st_attn_bwd_delta")
    return delta


def st_convert_f32(src, dtype=torch.bfloat16, out=None, stream=None):
    """fp32 tensor -> ``dtype`` (bf16 rounded to nearest even, or an fp32 copy)."""
    if out is None:
        out = torch.empty(src.shape, device=src.device, dtype=dtype)
    _check(load().st_convert_f32(src.numel(), _ptr(src), _ptr(out), _dtype_code(out.dtype), _stream(stream, out)),
           "st_convert_f32")
    return out


def st_fp16_scaled_copy(src, out=None, exps=None, scratch=None, stream=None):
    """Exact fp16 copy of a bf16 tensor scaled by 2^-e: returns (copy, e as a device int32 tensor)."""
    if out is None:
        out = torch.empty(src.shape, device=src.device, dtype=torch.float16)
    if exps is None:
        exps = torch.zeros(4, device=src.device, dtype=torch.int32)
    if scratch is None:
        scratch = torch.zeros(4, device=src.device, dtype=torch.int32)
    _check(load().st_fp16_scaled_copy(src.numel(), _ptr(src), _ptr(out), _ptr(exps), _ptr(scratch),
                                      _stream(stream, out, exps, scratch)), "st_fp16_scaled_copy")
    return out, exps
