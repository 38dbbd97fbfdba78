"""The N > 1 path of bench.py on the CPU (gloo, world size 2).

Every rank runs its own copy of the workload (weak scaling, no data-path
collective); the only cross-rank traffic is a barrier and the max over ranks of
the measured time.  These tests run that host logic in two processes.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    from domain_ring_attention_gb300.workloads import WORKLOADS, make_inputs
    r, w = bench.dist_init(world)
    assert (r, w) == (rank, world) and dist.get_backend() == "gloo"
    bench.barrier(w)
    slowest = bench.max_over_ranks(1.5 + rank, w)
    # each rank draws its own units of work (seed = rank), as the bench does
    qx, _, _ = make_inputs(WORKLOADS["tiny_fp32"], seed=r)
    t = qx.flatten()[:4].clone()
    gathered = [torch.zeros_like(t) for _ in range(w)]
    dist.all_gather(gathered, t)
    q.put((r, slowest, bool(torch.equal(gathered[0], gathered[1]))))
    dist.destroy_process_group()


def test_two_ranks_max_time_and_distinct_work():
    world, port = 2, free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert [r for r, _, _ in res] == [0, 1]
    assert all(s == 2.5 for _, s, _ in res)           # both ranks see the slowest rank's time
    assert not any(same for _, _, same in res)         # the two ranks' inputs differ


def test_reference_arm_under_torchrun_two_ranks():
    """`bench.py --impl reference` with two ranks: rank 0 times the oracle on
    the host cores and prints one JSON line; rank 1 exits without work."""
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--workload", "tiny_fp32", "--gpus", "2", "--steps", "1", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["unit"] == "TFLOP/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
