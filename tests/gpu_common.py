"""Shared helpers for the GPU parity tests (CUDA library vs float64 oracle).

Tolerances (stated for this method): fp32 inputs -- max abs error <= 1e-5;
bf16 inputs with fp32 accumulation -- max abs <= 1e-2 and mean abs <= 1e-3.
Gradients use the same bounds relative to the RMS of the oracle gradient.
"""
import numpy as np
import torch

import domain_ring_attention_gb300 as st
from domain_ring_attention_gb300.workloads import make_inputs
from oracle import attention as oa


def f64(t):
    return t.detach().float().cpu().double().numpy()


def assert_close(got, ref, dtype, name, rel_rms=False, scale=None):
    """Max and mean |got - ref| within the bound of `dtype`, relative to RMS(ref) with
    rel_rms.  `scale`: the RMS of a gradient of the same case that does not vanish
    (dV); when the exact gradient is zero (every query sees a single key: P = 1
    and dS = P (dP - Delta) = 0, so dQ = dK = 0), RMS(ref) is zero or float64
    rounding noise, and the error is measured on that scale instead."""
    err = np.abs(np.asarray(got, dtype=np.float64) - ref)
    den = float(np.sqrt(np.mean(ref * ref))) if rel_rms else 1.0
    if rel_rms and scale is not None and den < 1e-12 * scale:
        den = scale
    mx, mean = err.max() / den, err.mean() / den
    if dtype == "f32":
        assert mx <= 1e-5, "%s: max err %.3e > 1e-5" % (name, mx)
    else:
        assert mx <= 1e-2 and mean <= 1e-3, "%s: max %.3e mean %.3e" % (name, mx, mean)
    return mx, mean


def assert_lse(got, ref, dtype, name="lse"):
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), name + ": -inf pattern differs"
    assert_close(got[fin], ref[fin], dtype, name)


def run_case(wl, seed=0, backward=True, grad_dtype=torch.float32):
    """Forward (and backward) of one workload.

    For bf16 inputs the forward runs twice: with fp32 `out` (the value that is
    held to the tolerance) and with bf16 `out` (what the backward consumes),
    and the bf16 output must be the fp32 one rounded once.
    """
    q, k, v, do = (x.cuda() for x in make_inputs(wl, seed=seed, with_dout=True))
    lay = st.Layout(wl.lens, wl.zigzag)
    out, lse = st.st_attn_fwd(lay, q, k, v, causal=wl.causal)
    res = {"out": out, "lse": lse, "in": (q, k, v, do)}
    if q.dtype != torch.float32:
        out32, lse32 = st.st_attn_fwd(lay, q, k, v, causal=wl.causal, out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert torch.equal(out, out32.to(q.dtype)), "bf16 out is not the fp32 out rounded once"
        assert torch.equal(lse, lse32)
        res["out"], res["out_native"] = out32, out
    if backward:
        # the fp32 forward output gives Delta without the bf16 rounding of out
        res["grads"] = st.st_attn_bwd(lay, q, k, v, res["out"], lse, do, causal=wl.causal,
                                      grad_dtype=grad_dtype)
    torch.cuda.synchronize()
    assert_no_device_error()
    return res


def assert_no_device_error():
    rc = st.load().st_device_error(None)
    assert rc == 0, "device-side bounded wait gave up (%d)" % rc


def check_rows(wl, res, rows, heads):
    """Compare sampled rows of a large forward (rows are independent)."""
    qd, kd, vd = res["in"][:3]
    out, lse = f64(res["out"]), f64(res["lse"])
    for (b, h) in heads:
        qh = f64(qd[b:b + 1, :, h:h + 1])
        kh = f64(kd[b:b + 1, :, h:h + 1])
        vh = f64(vd[b:b + 1, :, h:h + 1])
        ro, rl = oa.forward_rows(qh, kh, vh, wl.lens, wl.zigzag, wl.causal, rows, heads=[(0, 0)])
        assert_close(out[b, rows, h], ro[(0, 0)], wl.dtype, "out[%d,%d]" % (b, h))
        assert_close(lse[b, h, rows], rl[(0, 0)], wl.dtype, "lse[%d,%d]" % (b, h))


def check_full(wl, res, backward=True):
    """Element-by-element comparison of a whole (small) case with the oracle."""
    q, k, v, do = (f64(x) for x in res["in"])
    ro, rl = oa.forward(q, k, v, wl.lens, wl.zigzag, wl.causal)
    assert_close(f64(res["out"]), ro, wl.dtype, "out")
    assert_lse(f64(res["lse"]), rl, wl.dtype)
    if backward:
        rg = oa.backward(q, k, v, ro, rl, do, wl.lens, wl.zigzag, wl.causal)
        dv_rms = float(np.sqrt(np.mean(rg[2] * rg[2])))
        for name, g, r in zip(("dq", "dk", "dv"), res["grads"], rg):
            assert_close(f64(g), r, wl.dtype, name, rel_rms=True, scale=dv_rms)


