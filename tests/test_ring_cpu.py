"""The multi-process ring schedule on the CPU (gloo; 2 and 3 ranks, one process each).

ShardTensor summary, section 4, ring attention: rank r keeps the queries of shard r while the K/V shards travel
round the ring; in training they travel with their dK/dV accumulators and return to their owner.  The schedule in
domain_ring_attention_gb300.ring runs here in separate processes with real point-to-point transfers (gloo), and
the arithmetic of each step is the oracle's (a block's partial merged by the log-sum-exp rule; a block's share
of the backward), so a block paired with the wrong shard, a step left out or an accumulator that does not come
home shows up as a difference from the oracle's unsharded attention and gradients.
"""
import math
import os
import socket
import sys
import types

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, lens, zigzag, causal, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    from domain_ring_attention_gb300 import ring
    from oracle import attention as oa
    from oracle import layout as ol
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        S, H, d = sum(lens), 2, 8
        g = np.random.default_rng(123)
        q, k, v, do = (g.standard_normal((1, S, H, d)) for _ in range(4))
        off, pos = ol.shard_offsets(lens), ol.natural_positions(lens, zigzag)
        mine = slice(off[rank], off[rank + 1])
        scale = 1 / math.sqrt(d)
        t64 = lambda x: torch.from_numpy(np.ascontiguousarray(x))
        lay = types.SimpleNamespace(D=world, lens=list(lens))
        seen = []

        def fwd_step(t, j, kb, vb, state):
            seen.append(j)
            o = np.zeros((1, off[rank + 1] - off[rank], H, d))
            l = np.zeros((1, H, off[rank + 1] - off[rank]))
            for h in range(H):
                o[0, :, h], l[0, h] = oa.partial_block(q[0, mine, h], kb.numpy()[0, :, h], vb.numpy()[0, :, h],
                                                       pos[mine], pos[off[j]:off[j + 1]], causal, scale)
                if state is not None:
                    o[0, :, h], l[0, h] = oa.merge_pair(state[0].numpy()[0, :, h], state[1].numpy()[0, h],
                                                        o[0, :, h], l[0, h])
            return t64(o), t64(l)

        out_r, lse_r = ring.ring_forward(lay, rank, t64(q[:, mine]), t64(k[:, mine]), t64(v[:, mine]),
                                         causal=causal, step=fwd_step)
        ref_o, ref_l = oa.forward(q, k, v, lens, zigzag, causal)
        ok_fwd = (np.allclose(out_r.numpy(), ref_o[:, mine], atol=1e-12)
                  and np.allclose(lse_r.numpy(), ref_l[:, :, mine], atol=1e-12))
        ring_order = seen == [(rank - t) % world for t in range(world)]

        delta = np.sum(do * ref_o, axis=3)                      # [1, S, H]

        def bwd_step(t, j, kb, vb, dk_acc, dv_acc, dq):
            ks = slice(off[j], off[j + 1])
            if t == 0:
                dq.zero_()
            for h in range(H):
                a, b, c = oa.block_grads(q[0, mine, h], kb.numpy()[0, :, h], vb.numpy()[0, :, h], do[0, mine, h],
                                         ref_l[0, h, mine], delta[0, mine, h], pos[mine], pos[ks], causal, scale)
                dq[0, :, h] += t64(a)
                dk_acc[0, :, h] += t64(b)
                dv_acc[0, :, h] += t64(c)

        qt, kt, vt = (t64(x[:, mine]) for x in (q, k, v))
        dq, dk, dv = ring.ring_backward(lay, rank, qt, kt, vt, None, None, None, causal=causal, step=bwd_step,
                                        acc_dtype=torch.float64)
        gq, gk, gv = oa.backward(q, k, v, ref_o, ref_l, do, lens, zigzag, causal)
        ok_bwd = all(np.allclose(mine_g.numpy(), ref[:, mine], atol=1e-12)
                     for mine_g, ref in ((dq, gq), (dk, gk), (dv, gv)))
        queue.put((rank, ok_fwd, ok_bwd, ring_order))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("lens,zigzag,causal", [((6, 10), True, True), ((5, 9, 3), False, False),
                                                ((4, 12, 2), True, True), ((2, 8, 4, 6), True, True)])
def test_ring_schedule_across_processes(lens, zigzag, causal):
    world, port = len(lens), free_port()
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, lens, zigzag, causal, queue)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    res = sorted(queue.get(timeout=10) for _ in range(world))
    assert [r[0] for r in res] == list(range(world))
    assert all(r[3] for r in res), "a rank did not meet the KV shards in ring order"
    assert all(r[1] for r in res), "forward differs from the oracle"
    assert all(r[2] for r in res), "backward differs from the oracle"
