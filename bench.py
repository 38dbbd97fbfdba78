"""Benchmark: sharded ring attention forward on one GB300 (and N replicas).

Default workload: ViT-style 4096^2 image, patch 16 -> S = 65536 tokens,
B=1, H=16, head_dim=64, bf16, D=16 equal shards, non-causal, forward only.
A step is one st_attn_fwd call (layout + ring-order fused forward with the
log-sum-exp merge) over inputs already resident in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

With N > 1 (torchrun, one rank per GPU) every rank runs the same workload on
its own GPU with no data-path collective (weak scaling); value = total FLOPs of
all ranks / the slowest rank's time.  ``--impl reference`` times the float64
CPU oracle on a bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np
import torch

from domain_ring_attention_gb300.workloads import WORKLOADS, make_inputs

METRIC = "ring-attention fwd/bwd TFLOP/s (bf16, S=65536) and % of GB300 dense-BF16 peak"
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
# dram bytes (read + write) of one full-size launch of the forward kernel on the
# default workload (16 heads), from the committed ncu capture of the kernel
# version named here; a kernel change without a new capture must drop its entry
# (traffic is then null).
NCU_TRAFFIC_BYTES = {"fwd_tc@6de3400": 423772672.0 + 123840000.0}
KERNEL_VERSION = "fwd_tc@6de3400"
DEFAULT_WORKLOAD = "vit4096_s65536"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--heads", type=int, default=None,
                   help="override H (a smaller capture of the same sequence shape for ncu)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--bwd", action="store_true",
                   help="time forward (fp32 out) + backward (fp32 gradients) as the step")
    p.add_argument("--no-train", action="store_true",
                   help="skip the secondary forward+backward measurement on train_s32768")
    return p.parse_args()


def dist_init(n):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:   # host-only runs (the reference arm's CPU oracle, CPU tests)
            dist.init_process_group("gloo")
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], device=dev, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            m = json.load(open(path))
            return (float(m.get("bf16_tflops")), float(m.get("bf16_tflops_sustained", m.get("bf16_tflops"))),
                    float(m.get("hbm_gbs")), "measured")
        except Exception:
            pass
    return FALLBACK_BF16_TFLOPS, 1700.0, FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        """Median SM clock, its maximum and the throttle reasons seen (computed
        once; later calls return the same result)."""
        if getattr(self, "_summary", None) is not None or self.proc is None:
            return getattr(self, "_summary", None)
        self.file.flush()
        rows = [l.strip().split(",") for l in open(self.file.name) if l.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[0]))
                mx = float(r[1])
                for name, val in zip(names, r[3:7]):
                    if "Active" in val and "Not" not in val:
                        reasons.add(name)
            except (ValueError, IndexError):
                continue
        if not sm:
            return None
        self._summary = {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                         "samples": len(sm)}
        return self._summary


def cpu_sample_tflops(wl, q, k, v, budget_s=12.0):
    """The float64 oracle on a bounded, growing sample of query rows."""
    from oracle import attention as oa
    rng = np.random.default_rng(0)
    S = wl.S
    heads = [(b, h) for b in range(wl.B) for h in range(wl.H)]
    flops = 0.0
    rows_done = 0
    t0 = time.perf_counter()
    it = 0
    while time.perf_counter() - t0 < budget_s:
        b, h = heads[it % len(heads)]
        rows = np.sort(rng.choice(S, size=min(64, S), replace=False))
        qh = q[b:b + 1, :, h:h + 1].float().numpy().astype(np.float64)
        kh = k[b:b + 1, :, h:h + 1].float().numpy().astype(np.float64)
        vh = v[b:b + 1, :, h:h + 1].float().numpy().astype(np.float64)
        oa.forward_rows(qh, kh, vh, wl.lens, wl.zigzag, wl.causal, rows, heads=[(0, 0)])
        vis = S if not wl.causal else (S + 1) / 2.0
        flops += 4.0 * wl.d * vis * len(rows)
        rows_done += len(rows)
        it += 1
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return flops / dt / 1e12, rows_done, dt, cores


# ex2 results per clock per SM, measured on GB300 (ex2.approx.ftz.f32 throughput
# probe: 30.5 per clock per SM with every warp issuing only exponentials)
MUFU_EX2_PER_CLK_SM = 30.5
GB300_SMS = 152


def cool_down(seconds=1.0):
    """Free cached blocks and let the GPU idle before the next secondary
    measurement (outside every timed region)."""
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    time.sleep(seconds)


def merge_gbs(st, wl, world, steps=10, warmup=3):
    """Standalone log-sum-exp merge (st_attn_merge) of D per-KV-shard partials
    of the workload's shape: HBM-bound, reported as algorithmic GB/s (partials
    and their lse read once, out in bf16 and lse written once).  Inputs are
    random partials (the merge's cost does not depend on their values) and far
    larger than L2."""
    dev = torch.device("cuda", torch.cuda.current_device())
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    po = torch.randn((wl.D, wl.B, wl.S, wl.H, wl.d), device=dev, dtype=torch.float32, generator=g)
    pl = torch.randn((wl.D, wl.B, wl.H, wl.S), device=dev, dtype=torch.float32, generator=g)
    out = torch.empty((wl.B, wl.S, wl.H, wl.d), device=dev, dtype=torch.bfloat16)
    lse = torch.empty((wl.B, wl.H, wl.S), device=dev, dtype=torch.float32)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        st.st_attn_merge(po, pl, out=out, lse=lse, stream=stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        st.st_attn_merge(po, pl, out=out, lse=lse, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / steps, world)
    nbytes = po.numel() * 4 + pl.numel() * 4 + out.numel() * 2 + lse.numel() * 4
    _, _, hbm, kind = peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    del po, pl
    return {"kernel": "merge_kernel (st_attn_merge)", "D": wl.D, "bytes_per_launch": nbytes, "ms": ms,
            "achieved_gbs": gbs, "peak_gbs": hbm, "frac": gbs / hbm, "peak_kind": kind + " HBM copy"}


def hbm_steps_gbs(st, world, steps=10, warmup=3):
    """The backward's bandwidth-bound steps on their own, at the training
    workload's shapes (B=2, S=32768, H=32, d=128): Delta = rowsum(dO o O)
    (st_attn_bwd_delta: fp32 out and bf16 dO read, 4 B per row written), the
    fp32 -> bf16 conversion of the dQ accumulator (st_convert_f32: 4 B read,
    2 B written per element) and the exact fp16 operand copy of one bf16
    tensor (st_fp16_scaled_copy: its max pass and its copy pass read the
    tensor twice and write the copy once, 6 B per element).  Each is
    reported as its bytes / CUDA-event time against the measured HBM copy;
    the tensors (0.5-1 GiB each) exceed L2."""
    from domain_ring_attention_gb300 import _lib
    wl = WORKLOADS["train_s32768"]
    dev = torch.device("cuda", torch.cuda.current_device())
    g = torch.Generator(device=dev)
    g.manual_seed(29)
    shape = (wl.B, wl.S, wl.H, wl.d)
    n = wl.B * wl.S * wl.H * wl.d
    out32 = torch.randn(shape, device=dev, generator=g)
    do16 = torch.randn(shape, device=dev, generator=g).to(torch.bfloat16)
    delta = torch.empty((wl.B, wl.H, wl.S), device=dev)
    dst16 = torch.empty(shape, device=dev, dtype=torch.bfloat16)
    h16 = torch.empty(shape, device=dev, dtype=torch.float16)
    exps = torch.zeros(4, device=dev, dtype=torch.int32)
    scratch = torch.zeros(4, device=dev, dtype=torch.int32)
    stream = torch.cuda.current_stream()
    jobs = {
        "delta": (lambda: _lib.st_attn_bwd_delta(out32, do16, delta=delta, stream=stream),
                  n * 4 + n * 2 + wl.B * wl.H * wl.S * 4, "delta_kernel (st_attn_bwd_delta)", 1),
        "convert": (lambda: _lib.st_convert_f32(out32, torch.bfloat16, out=dst16, stream=stream),
                    n * 4 + n * 2, "convert_kernel (st_convert_f32)", 1),
        "fp16_copy": (lambda: _lib.st_fp16_scaled_copy(do16, out=h16, exps=exps, scratch=scratch, stream=stream),
                      n * 2 * 2 + n * 2, "amax_kernel + fp16_copy_kernel (st_fp16_scaled_copy)", 2),
    }
    _, _, hbm, kind = peaks()
    res = {}
    for name, (fn, nbytes, kernel, launches) in jobs.items():
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = max_over_ranks(e0.elapsed_time(e1) / steps, world)
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[name] = {"kernel": kernel, "bytes_per_call": nbytes, "ms": ms, "achieved_gbs": gbs, "peak_gbs": hbm,
                     "frac": gbs / hbm, "peak_kind": kind + " HBM copy", "launches": launches}
    return res


def proj_tflops(st, wl, world, steps=10, warmup=3):
    """The projections on either side of the attention for the workload's
    shape (st_proj_gemm, bf16 in, fp32 accumulation, bf16 out): the packed
    QKV input projection [B*S, H*d] x [3*H*d, H*d]^T and the output
    projection [B*S, H*d] x [H*d, H*d]^T, random weights."""
    dev = torch.device("cuda", torch.cuda.current_device())
    g = torch.Generator(device=dev)
    g.manual_seed(13)
    hidden = wl.H * wl.d
    M = wl.B * wl.S
    x = torch.randn((M, hidden), device=dev, generator=g).to(torch.bfloat16)
    res = {}
    for name, n_out in (("qkv", 3 * hidden), ("out", hidden)):
        w = (torch.randn((n_out, hidden), device=dev, generator=g) / hidden ** 0.5).to(torch.bfloat16)
        y = torch.empty((M, n_out), device=dev, dtype=torch.bfloat16)
        stream = torch.cuda.current_stream()
        for _ in range(warmup):
            st.st_proj_gemm(x, w, out=y, stream=stream)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            st.st_proj_gemm(x, w, out=y, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        ms = max_over_ranks(e0.elapsed_time(e1) / steps, world)
        peak_b, _, _, kind = peaks()
        tf = 2.0 * M * n_out * hidden / (ms * 1e-3) / 1e12
        res[name] = {"M": M, "N": n_out, "K": hidden, "ms": ms, "tflops": tf, "frac": tf / peak_b,
                     "peak_kind": kind + " burst bf16"}
    return res


def mlp_tflops(st, world, steps=10, warmup=3):
    """The gated MLP that TSP pairs with its ring schedule (st_gated_mlp: the
    gate and up GEMM with the SiLU-gated epilogue, then the down GEMM), at the
    7B-style width (hidden 4096 = 32 heads x 128, F = 11008) over 65536 tokens,
    random weights; 6*M*hidden*F flops per call."""
    dev = torch.device("cuda", torch.cuda.current_device())
    g = torch.Generator(device=dev)
    g.manual_seed(17)
    M, hidden, F = 65536, 4096, 11008
    x = torch.randn((M, hidden), device=dev, generator=g).to(torch.bfloat16)
    w1 = (torch.randn((F, hidden), device=dev, generator=g) / hidden ** 0.5).to(torch.bfloat16)
    w3 = (torch.randn((F, hidden), device=dev, generator=g) / hidden ** 0.5).to(torch.bfloat16)
    w2 = (torch.randn((hidden, F), device=dev, generator=g) / F ** 0.5).to(torch.bfloat16)
    h = torch.empty((M, F), device=dev, dtype=torch.bfloat16)
    y = torch.empty((M, hidden), device=dev, dtype=torch.bfloat16)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        st.st_gated_mlp(x, w1, w3, w2, out=y, h=h, stream=stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        st.st_gated_mlp(x, w1, w3, w2, out=y, h=h, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / steps, world)
    peak_b, _, _, kind = peaks()
    tf = 6.0 * M * hidden * F / (ms * 1e-3) / 1e12
    return {"M": M, "hidden": hidden, "F": F, "ms": ms, "tflops": tf, "frac": tf / peak_b,
            "peak_kind": kind + " burst bf16", "launches": 2}


def conv_tflops(st, world, steps=10, warmup=3):
    """Halo exchange + 2-D convolution of a row-sharded image (st_halo_exchange
    then st_conv2d_sharded): the CONUS grid 1024 x 1792, 256 channels in and
    out, 3 x 3 kernel, D = 4 Dirichlet-uneven row shards, bf16 in and out,
    random weights.  2*H*W*C_in*C_out*k*k flops per step; the inputs (0.94 GB)
    and outputs exceed L2."""
    from domain_ring_attention_gb300.workloads import dirichlet_shard_lengths
    dev = torch.device("cuda", torch.cuda.current_device())
    g = torch.Generator(device=dev)
    g.manual_seed(19)
    H, W, C, k = 1024, 1792, 256, 3
    rows = dirichlet_shard_lengths(H, 4, seed=0, multiple=1)
    shards = [torch.randn((L + 2, W, C), device=dev, generator=g).to(torch.bfloat16) for L in rows]
    w = (torch.randn((C, k, k, C), device=dev, generator=g) / (k * k * C) ** 0.5).to(torch.bfloat16)
    b = torch.zeros((C,), device=dev)
    out = [torch.empty((L, W, C), device=dev, dtype=torch.bfloat16) for L in rows]
    stream = torch.cuda.current_stream()

    def step():
        st.st_halo_exchange(shards, 1, stream=stream)
        st.st_conv2d_sharded(shards, w, b, out=out, stream=stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / steps, world)
    peak_b, _, _, kind = peaks()
    tf = 2.0 * H * W * C * C * k * k / (ms * 1e-3) / 1e12
    return {"H": H, "W": W, "C_in": C, "C_out": C, "k": k, "shard_rows": rows, "ms": ms, "tflops": tf,
            "frac": tf / peak_b, "peak_kind": kind + " burst bf16", "launches": 2}


def norm_gbs(st, world, steps=10, warmup=3):
    """Group normalisation of the row-sharded CONUS grid (st_group_norm_sharded:
    statistics, their all-reduce over the shards, normalisation): 1024 x 1792
    pixels, 256 channels in 32 groups, four Dirichlet-uneven row shards, bf16
    in and out.  HBM-bound, reported as algorithmic GB/s: the statistics need
    every value before the first output, so x is read twice and y written
    once (3 x 0.94 GB); x exceeds L2."""
    from domain_ring_attention_gb300.workloads import dirichlet_shard_lengths
    dev = torch.device("cuda", torch.cuda.current_device())
    g = torch.Generator(device=dev)
    g.manual_seed(23)
    H, W, C, G = 1024, 1792, 256, 32
    rows = dirichlet_shard_lengths(H, 4, seed=0, multiple=1)
    xs = [torch.randn((L, W, C), device=dev, generator=g).to(torch.bfloat16) for L in rows]
    out = [torch.empty((L, W, C), device=dev, dtype=torch.bfloat16) for L in rows]
    gamma = torch.ones(C, device=dev)
    beta = torch.zeros(C, device=dev)
    ws = torch.empty(1 << 20, device=dev, dtype=torch.uint8)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        st.st_group_norm_sharded(xs, G, gamma, beta, out=out, workspace=ws, stream=stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        st.st_group_norm_sharded(xs, G, gamma, beta, out=out, workspace=ws, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / steps, world)
    nbytes = 3 * H * W * C * 2
    _, _, hbm, kind = peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"H": H, "W": W, "C": C, "G": G, "shard_rows": rows, "bytes_per_step": nbytes, "ms": ms,
            "achieved_gbs": gbs, "peak_gbs": hbm, "frac": gbs / hbm, "peak_kind": kind + " HBM copy", "launches": 3}


def train_step_tflops(st, world, steps=3, warmup=2, name="train_s32768"):
    """Forward + backward on a workload: the training workload (B=2, H=32,
    d=128, S=32768, causal zigzag over Dirichlet sharding shapes), the 7B-style
    one (B=1, H=32, d=128, S=131072, 8 equal shards = 16 zigzag chunks) or the
    ViT 1024^2 one (B=1, H=16, d=64, S=4096, 8 shards, non-causal).  One step =
    st_attn_fwd (fp32 out) + st_attn_bwd (fp32 gradients), inputs resident in
    HBM (the ViT 1024^2 inputs, 24 MiB, stay in L2 between steps)."""
    wl = WORKLOADS[name]
    dev = torch.device("cuda", torch.cuda.current_device())
    q, k, v, do = make_inputs(wl, seed=7, device=dev, with_dout=True)
    lay = st.Layout(wl.lens, wl.zigzag)
    out = torch.empty(q.shape, device=dev, dtype=torch.float32)
    lse = torch.empty((wl.B, wl.H, wl.S), device=dev, dtype=torch.float32)
    wsf = torch.empty(st.st_attn_workspace_size(lay, wl.B, wl.H, wl.d, q.dtype, 0), device=dev,
                      dtype=torch.uint8)
    wsb = torch.empty(st.st_attn_workspace_size(lay, wl.B, wl.H, wl.d, q.dtype, 1), device=dev,
                      dtype=torch.uint8)
    stream = torch.cuda.current_stream()

    def fwd():
        st.st_attn_fwd(lay, q, k, v, causal=wl.causal, out=out, lse=lse, stream=stream, workspace=wsf)

    def bwd():
        st.st_attn_bwd(lay, q, k, v, out, lse, do, causal=wl.causal, workspace=wsb, stream=stream)

    for _ in range(warmup):
        fwd()
        bwd()
    torch.cuda.synchronize()
    barrier(world)
    # the steps are queued back to back, as a training loop queues them (the host
    # runs ahead of the GPU), with events around each pass, read after one
    # synchronize; a small problem is then not charged the host's launch latency
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for e in ev:
        e[0].record(stream)
        fwd()
        e[1].record(stream)
        bwd()
        e[2].record(stream)
    torch.cuda.synchronize()
    tf = sum(e[0].elapsed_time(e[1]) for e in ev)
    tb = sum(e[1].elapsed_time(e[2]) for e in ev)
    tf = max_over_ranks(tf / steps, world)
    tb = max_over_ranks(tb / steps, world)
    res = {"workload": name, "shard_lens": list(wl.lens), "causal": wl.causal, "zigzag": wl.zigzag,
            "fwd_tflops": wl.fwd_flops() * world / (tf * 1e-3) / 1e12,
            "bwd_tflops": wl.bwd_flops() * world / (tb * 1e-3) / 1e12,
            "fwd_bwd_tflops": (wl.fwd_flops() + wl.bwd_flops()) * world / ((tf + tb) * 1e-3) / 1e12,
            "fwd_ms": tf, "bwd_ms": tb,
            "note": "fwd writes fp32 out (the backward's Delta); bwd writes fp32 dq, dk, dv"}
    peak_b, _, _, kind = peaks()
    for key in ("fwd", "bwd", "fwd_bwd"):
        res[key + "_frac"] = res[key + "_tflops"] / world / peak_b
    res["peak_tflops"] = peak_b
    res["peak_kind"] = kind + " burst bf16 (fractions per GPU)"
    return res


def ring_local_tflops(st, world, steps=3, warmup=2, name="train_s32768"):
    """The ring schedule with every rank's shard on this one GPU (st_ring_fwd_local /
    st_ring_bwd_local): rank r keeps query shard r, the K/V blocks (in the
    backward with their dK/dV accumulators) pass from rank to rank by device
    copies on a second stream while the previous blocks compute.  On one GPU the
    D ranks' step kernels run one after another, so this measures the ring's
    per-step kernels and copies, not a multi-GPU ring; the fused kernels are the
    one-GPU path.  fp32 outputs and gradients."""
    from domain_ring_attention_gb300 import _lib
    wl = WORKLOADS[name]
    dev = torch.device("cuda", torch.cuda.current_device())
    q, k, v, do = make_inputs(wl, seed=9, device=dev, with_dout=True)
    lay = st.Layout(wl.lens, wl.zigzag)
    off = np.cumsum([0] + list(wl.lens))
    cut = lambda x: [x[:, off[r]:off[r + 1]].contiguous() for r in range(wl.D)]
    qs, ks, vs, dos = cut(q), cut(k), cut(v), cut(do)
    del q, k, v, do
    wsf = torch.empty(_lib.st_ring_workspace_size(lay, wl.B, wl.H, wl.d, 2), device=dev, dtype=torch.uint8)
    wsb = torch.empty(_lib.st_ring_workspace_size(lay, wl.B, wl.H, wl.d, 3), device=dev, dtype=torch.uint8)
    stream = torch.cuda.current_stream()
    copy_stream = torch.cuda.Stream()
    state = {}

    def fwd():
        state["o"], state["l"] = _lib.st_ring_fwd_local(lay, qs, ks, vs, causal=wl.causal, out_dtype=torch.float32,
                                                        stream=stream, copy_stream=copy_stream, workspace=wsf)

    def bwd():
        _lib.st_ring_bwd_local(lay, qs, ks, vs, state["o"], state["l"], dos, causal=wl.causal, stream=stream,
                               copy_stream=copy_stream, workspace=wsb)

    for _ in range(warmup):
        fwd()
        bwd()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    tf = tb = 0.0
    for _ in range(steps):
        ev[0].record(stream)
        fwd()
        ev[1].record(stream)
        bwd()
        ev[2].record(stream)
        torch.cuda.synchronize()
        tf += ev[0].elapsed_time(ev[1])
        tb += ev[1].elapsed_time(ev[2])
    tf = max_over_ranks(tf / steps, world)
    tb = max_over_ranks(tb / steps, world)
    return {"workload": name, "ranks_on_one_gpu": wl.D, "fwd_tflops": wl.fwd_flops() / (tf * 1e-3) / 1e12,
            "bwd_tflops": wl.bwd_flops() / (tb * 1e-3) / 1e12, "fwd_ms": tf, "bwd_ms": tb,
            "note": "ring schedule emulated on one GPU: the D ranks' step kernels run one after another"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    wl = WORKLOADS[args.workload]
    g = torch.Generator().manual_seed(0)
    shape = (wl.B, wl.S, wl.H, wl.d)
    q, k, v = (torch.randn(shape, generator=g).to(wl.torch_dtype) for _ in range(3))
    vals = []
    info = None
    for i in range(args.warmup + args.steps):
        val, rows, dt, cores = cpu_sample_tflops(wl, q, k, v, budget_s=2.0)
        if i >= args.warmup:
            vals.append(val)
            info = (rows, dt, cores)
    value = statistics.median(vals)
    sample = "%d query rows per step over all heads, float64 numpy oracle" % info[0]
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": info[1] * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(wl.describe(), parallelism="replicas%d" % world),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": info[2], "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world):
    import domain_ring_attention_gb300 as st
    st.load()
    wl = WORKLOADS[args.workload]
    if args.heads:
        import dataclasses
        wl = dataclasses.replace(wl, H=args.heads)
    dev = torch.device("cuda", torch.cuda.current_device())
    q_h, k_h, v_h = make_inputs(wl, seed=rank, device="cpu")
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    lay = st.Layout(wl.lens, wl.zigzag)
    out = torch.empty(q.shape, device=dev, dtype=torch.float32 if args.bwd else q.dtype)
    lse = torch.empty((wl.B, wl.H, wl.S), device=dev, dtype=torch.float32)
    ws = torch.empty(max(1, st.st_attn_workspace_size(lay, wl.B, wl.H, wl.d, q.dtype, 0)),
                     device=dev, dtype=torch.uint8)
    stream = torch.cuda.current_stream()
    # kernels of one forward step: bf16 -> max|v|, fp16 copy of v, fused forward
    launches_per_step = 3 if q.dtype == torch.bfloat16 else 1
    flops = wl.fwd_flops()
    if args.bwd:
        do = make_inputs(wl, seed=1000 + rank, device=dev, with_dout=True)[3]
        wsb = torch.empty(st.st_attn_workspace_size(lay, wl.B, wl.H, wl.d, q.dtype, 1), device=dev,
                          dtype=torch.uint8)
        flops += wl.bwd_flops()
        # backward: Delta, max|x| of four tensors, their fp16 copies, the fused backward
        launches_per_step += 4 if q.dtype == torch.bfloat16 else 2

    def step():
        st.st_attn_fwd(lay, q, k, v, causal=wl.causal, out=out, lse=lse, stream=stream, workspace=ws)
        if args.bwd:
            st.st_attn_bwd(lay, q, k, v, out, lse, do, causal=wl.causal, workspace=wsb, stream=stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(torch.cuda.current_device()) as clk:
        time.sleep(0.3)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(args.steps):
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        t1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    total_ms = max_over_ranks(t0.elapsed_time(t1), world)
    launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms_per_step = total_ms / args.steps
    value = flops * world / (ms_per_step * 1e-3) / 1e12
    peak_b, peak_s, hbm, peak_kind = peaks()
    achieved = flops / (statistics.mean(launch_ms) * 1e-3) / 1e12

    # exponentials: one per visible pair; against the MUFU rate measured on GB300
    n_exp = wl.fwd_flops() / (4 * wl.d)
    mufu = None
    if not args.bwd:
        clk_mhz = (clk.summary() or {}).get("sm_mhz") or 2070.0
        peak_exp = MUFU_EX2_PER_CLK_SM * GB300_SMS * clk_mhz * 1e6
        exps = n_exp / (statistics.mean(launch_ms) * 1e-3)
        mufu = {"exps_per_s": exps, "peak_exps_per_s": peak_exp, "frac": exps / peak_exp,
                "peak_kind": "measured ex2 throughput x 152 SMs x SM clock"}
    e2e = None
    if not args.no_e2e:
        pin = [x.pin_memory() for x in (q_h, k_h, v_h)]
        out_h = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        lse_h = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
        qd, kd, vd = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        copy_stream = torch.cuda.Stream()
        dev = {"q": qd, "k": kd, "v": vd, "out": out, "lse": lse}

        def e2e_step():
            if out.dtype == torch.bfloat16:
                # the host-buffer entry point: heads in groups, each group's copies
                # in, compute and copies back overlapped with the other groups'
                st.st_attn_fwd_host(lay, pin[0], pin[1], pin[2], out_h, lse_h, dev, causal=wl.causal,
                                    workspace=ws, stream=stream, copy_stream=copy_stream)
                return
            qd.copy_(pin[0], non_blocking=True)
            kd.copy_(pin[1], non_blocking=True)
            vd.copy_(pin[2], non_blocking=True)
            st.st_attn_fwd(lay, qd, kd, vd, causal=wl.causal, out=out, lse=lse, stream=stream,
                           workspace=ws)
            out_h.copy_(out, non_blocking=True)
            lse_h.copy_(lse, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        n_e2e = max(3, min(args.steps, 10))
        e0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(e0.elapsed_time(e1) / n_e2e, world)
        h2d = sum(x.numel() * x.element_size() for x in pin)
        d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()
        e2e = {"value": flops * world / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms}

    # the secondary kernels after the end-to-end run, each after a pause so
    # that none starts under the power cap that the previous one ran into;
    # the gated MLP, which draws the most, goes last
    merge = proj = mlp = conv = gnorm = hbm_steps = None
    if not args.no_train and world == 1 and not args.bwd:
        cool_down()
        merge = merge_gbs(st, wl, world)
        cool_down()
        hbm_steps = hbm_steps_gbs(st, world)
        cool_down()
        proj = proj_tflops(st, wl, world)
        cool_down()
        conv = conv_tflops(st, world)
        cool_down()
        gnorm = norm_gbs(st, world)
        cool_down()
        mlp = mlp_tflops(st, world)
        cool_down()

    if not args.no_train:
        cool_down()
    train = None if args.no_train else train_step_tflops(st, world)
    llm7b = ring_local = None
    if not args.no_train and not args.bwd:
        cool_down()
        llm7b = train_step_tflops(st, world, name="llm7b_causal_s131072")
        if world == 1:
            cool_down()
            ring_local = ring_local_tflops(st, world)
    vit1024 = None
    if not args.no_train and not args.bwd and world == 1:
        cool_down()
        vit1024 = train_step_tflops(st, world, steps=20, warmup=5, name="vit1024_s4096")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        val, rows, dt, cores = cpu_sample_tflops(wl, q_h, k_h, v_h, budget_s=12.0)
        cpu = {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": "%d query rows (64 per head, cycling heads) of the same workload, "
                         "float64 numpy, %.1f s" % (rows, dt)}

    if rank == 0:
        in_bytes = 3 * q.numel() * q.element_size()
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": dict(wl.describe(), parallelism="replicas%d" % world,
                           l2=("inputs %d MiB > 129 MB L2, no flush" % (in_bytes >> 20) if in_bytes > 129e6 else
                               "inputs %d MiB fit in the 129 MB L2 and stay there between steps (no flush)"
                               % (in_bytes >> 20))),
            "pct_of_peak": 100.0 * value / world / peak_b,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_b,
                         "unit": "TFLOP/s", "frac": achieved / peak_b,
                         # the recorded capture is of the default forward workload only
                         "traffic": (NCU_TRAFFIC_BYTES.get(KERNEL_VERSION)
                                     if args.workload == DEFAULT_WORKLOAD and not args.bwd and not args.heads
                                     else None),
                         "peak_kind": peak_kind + " burst bf16"},
            "gpu_launches": args.steps * launches_per_step,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "clocks": clk.summary(),
            "secondary": {"train": train, "llm7b": llm7b, "vit1024": vit1024, "ring_local": ring_local, "merge": merge, "bwd_hbm_steps": hbm_steps, "mufu": mufu, "proj": proj, "mlp": mlp, "conv": conv, "norm": gnorm},
        }
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, world = dist_init(args.gpus)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
