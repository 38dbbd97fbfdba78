"""Ring attention across processes: one rank per GPU, K/V shards passed round the ring.

ShardTensor summary, section 4, ring attention: the sequence is split into D shards of any lengths (the sharding
shapes of section 2), rank r keeps the queries of shard r, and the K/V shards travel round a ring of ranks.  At
step t rank r holds the K/V of shard (r - t) mod D: it computes that shard's partial result for its queries while
it already sends the block on to rank r + 1 and receives the next one from rank r - 1, and it folds the partial
into its running result by the log-sum-exp rule.  In training the K/V shards travel with their dK/dV
accumulators, every rank adds its queries' block to them, and one more hop after the last step brings them home.

This module is the schedule only: which block is where at every step, and the transfers, carried by
torch.distributed (NCCL between GPUs; gloo for host-only tests).  The arithmetic of a step is a call of the C-ABI
library (st_ring_fwd_step, st_ring_bwd_step); ``step`` arguments replace it, e.g. in host-only tests.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import _lib


def _exchange(send, recv_shapes, rank, world, group=None):
    """Send the tensors ``send`` to rank + 1 and receive tensors of ``recv_shapes`` (shape, dtype) from rank - 1,
    all in one batch of point-to-point operations.  Returns (received tensors, requests)."""
    nxt, prv = (rank + 1) % world, (rank - 1) % world
    device = send[0].device
    recv = [torch.empty(s, dtype=dt, device=device) for s, dt in recv_shapes]
    ops = [dist.P2POp(dist.isend, t, nxt, group) for t in send]
    ops += [dist.P2POp(dist.irecv, t, prv, group) for t in recv]
    return recv, dist.batch_isend_irecv(ops)


def _block_shape(t, rows):
    return (int(t.shape[0]), int(rows)) + tuple(int(x) for x in t.shape[2:])


def ring_forward(layout, rank, q, k, v, causal=False, scale=0.0, step=None, group=None):
    """Ring attention forward on rank ``rank`` of D = layout.D ranks.

    q, k, v: the rank's shard, [B, L_rank, H, d] (bf16 for the library's step).  ``step(t, kv_shard, k_blk,
    v_blk, state) -> state`` folds one held block into the running state (None before the first step); the
    default is the library's st_ring_fwd_step with an fp32 running (out, lse).  Returns the final state.
    """
    world = layout.D
    if dist.is_initialized() and dist.get_world_size(group) != world:
        raise ValueError("one rank per shard: the group has %d ranks, the layout %d shards"
                         % (dist.get_world_size(group), world))
    if step is None:
        ws = torch.empty(_lib.st_ring_workspace_size(layout, int(q.shape[0]), int(q.shape[2]), int(q.shape[3]), 0),
                         device=q.device, dtype=torch.uint8)

        def step(t, j, kb, vb, state):
            out = state[0] if state is not None else None
            lse = state[1] if state is not None else None
            return _lib.st_ring_fwd_step(layout, rank, j, q, kb, vb, prev=state, causal=causal, scale=scale,
                                         out=out, lse=lse, workspace=ws)

    held_k, held_v = k, v
    state = None
    for t in range(world):
        j = (rank - t) % world
        reqs = []
        if t + 1 < world:
            # the block rank - 1 holds at this step travels here while this step computes
            j_in = (rank - 1 - t) % world
            shape = _block_shape(k, layout.lens[j_in])
            (nk, nv), reqs = _exchange([held_k, held_v], [(shape, k.dtype), (shape, v.dtype)], rank, world, group)
        state = step(t, j, held_k, held_v, state)
        for r in reqs:
            r.wait()
        if t + 1 < world:
            held_k, held_v = nk, nv
    return state


def ring_backward(layout, rank, q, k, v, out, lse, dout, causal=False, scale=0.0, step=None, group=None,
                  acc_dtype=torch.float32):
    """Ring attention backward on rank ``rank``: returns fp32 (dq, dk, dv) of the rank's shard.

    K and V pass on while a step computes; the fp32 dK/dV accumulators of the held shard pass on after the step
    has added to them, and after the last step they travel one more hop, to the shard's owner.  ``step(t,
    kv_shard, k_blk, v_blk, dk_acc, dv_acc, dq)`` adds one block's contributions in place (dq zeroed by the
    first step); the default is the library's st_ring_bwd_step, whose accumulators are fp32 (``acc_dtype``).
    """
    world = layout.D
    B, L, H, d = (int(x) for x in q.shape)
    if step is None:
        ws = torch.empty(_lib.st_ring_workspace_size(layout, B, H, d, 1), device=q.device, dtype=torch.uint8)

        def step(t, j, kb, vb, dk_acc, dv_acc, dq_):
            _lib.st_ring_bwd_step(layout, rank, j, q, kb, vb, out, lse, dout, dq_, dk_acc, dv_acc, t == 0,
                                  causal=causal, scale=scale, workspace=ws)

    dq = torch.zeros((B, L, H, d), dtype=acc_dtype, device=q.device)
    held_k, held_v = k, v
    acc_k = torch.zeros((B, L, H, d), dtype=acc_dtype, device=q.device)
    acc_v = torch.zeros_like(acc_k)
    for t in range(world):
        j = (rank - t) % world
        j_in = (rank - 1 - t) % world
        shape_in = _block_shape(k, layout.lens[j_in])
        kv_reqs = []
        if t + 1 < world:
            (nk, nv), kv_reqs = _exchange([held_k, held_v], [(shape_in, k.dtype), (shape_in, v.dtype)], rank,
                                          world, group)
        step(t, j, held_k, held_v, acc_k, acc_v, dq)
        if world == 1:
            break
        # the accumulators move on once this step has added to them; after the last step this is the hop home
        (ak, av), acc_reqs = _exchange([acc_k, acc_v], [(shape_in, acc_dtype), (shape_in, acc_dtype)], rank, world,
                                       group)
        for r in kv_reqs + acc_reqs:
            r.wait()
        acc_k, acc_v = ak, av
        if t + 1 < world:
            held_k, held_v = nk, nv
    # after D hops the accumulators of this rank's own shard are back
    return dq, acc_k, acc_v
