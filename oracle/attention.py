"""Oracle attention: definition, ring formulation with log-sum-exp merge, backward.

Test infrastructure only (see the package docstring).  float64 throughout;
numpy matmul is the only library step.  Tensors are BSHD ``[B, S, H, d]`` in
buffer ("sharded") order; ``lse`` is ``[B, H, S]`` (natural log).

Definition (ShardTensor summary, section 4: ring attention is benchmarked as
the domain-parallel form of ordinary attention, and domain-parallel results
must stay numerically consistent with the unsharded computation, section 2
"communication"; TSP summary, section 2: K/V are all-gathered and
FlashAttention computes plain attention over them):

    s_ij   = scale * <q_i, k_j>             over visible pairs (i, j)
    lse_i  = log sum_j exp(s_ij)
    out_i  = sum_j exp(s_ij - lse_i) v_j

with scale = 1/sqrt(d) unless given (the pages print no scale; this is the
usual softmax(QK^T/sqrt(d))V reading).  Visible means every j when not causal;
when causal, pos[j] <= pos[i] in *natural* sequence positions (the zigzag
re-partition moves rows in the buffer but not in the sequence).

Ring formulation: each query shard r meets every KV shard j in turn and forms
a partial (O_rj, lse_rj) over the keys of shard j only; partials are combined
by the log-sum-exp rule (``merge_pair``).  A partial with no visible key has
lse = -inf and O = 0, and is the identity of the merge.

Backward (the textbook gradient of the definition): with P_ij = exp(s_ij -
lse_i) on visible pairs,
    dV_j = sum_i P_ij dO_i,   dP_ij = <dO_i, v_j>,   Delta_i = <dO_i, out_i>,
    dS_ij = P_ij (dP_ij - Delta_i),
    dQ_i = scale sum_j dS_ij k_j,   dK_j = scale sum_i dS_ij q_i.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from .layout import natural_positions, shard_offsets

NEG_INF = -np.inf


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


def _as_f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def _row_block(S: int) -> int:
    return int(max(16, min(1024, (1 << 24) // max(S, 1))))


def _softmax_rows(s: np.ndarray):
    """Row-wise (lse, P) of a score block whose masked entries are -inf.

    A row with no finite score gets lse = -inf and P = 0.
    """
    m = np.max(s, axis=1)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    e = np.exp(s - m_safe[:, None])          # exp(-inf) = 0 for masked entries
    tot = np.sum(e, axis=1)
    with np.errstate(divide="ignore"):
        lse = np.where(finite, m_safe + np.log(np.where(finite, tot, 1.0)), NEG_INF)
    p = np.where(finite[:, None], e / np.where(finite, tot, 1.0)[:, None], 0.0)
    return lse, p


def _visible(qpos: np.ndarray, kpos: np.ndarray, causal: bool) -> np.ndarray:
    if not causal:
        return np.ones((qpos.size, kpos.size), dtype=bool)
    return kpos[None, :] <= qpos[:, None]


def forward(q, k, v, lens, zigzag=False, causal=False, scale=None):
    """Full attention of every buffer row.  Returns (out [B,S,H,d], lse [B,H,S])."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, S, H, d = q.shape
    if scale is None:
        scale = default_scale(d)
    pos = natural_positions(lens, zigzag)
    if pos.size != S:
        raise ValueError("sharding shapes do not add up to S")
    order = np.argsort(pos, kind="stable")   # natural position -> buffer row
    out = np.zeros_like(q)
    lse = np.zeros((B, H, S))
    blk = _row_block(S)
    for b in range(B):
        for h in range(H):
            qn = q[b, order, h, :]
            kn = k[b, order, h, :]
            vn = v[b, order, h, :]
            for i0 in range(0, S, blk):
                i1 = min(S, i0 + blk)
                s = scale * (qn[i0:i1] @ kn.T)
                if causal:   # natural order: key j visible to query i iff j <= i
                    rows = np.arange(i0, i1)[:, None]
                    s = np.where(np.arange(S)[None, :] <= rows, s, NEG_INF)
                l_blk, p = _softmax_rows(s)
                out[b, order[i0:i1], h, :] = p @ vn
                lse[b, h, order[i0:i1]] = l_blk
    return out, lse


def forward_rows(q, k, v, lens, zigzag, causal, rows, scale=None, heads=None):
    """Attention of selected buffer rows only (rows are independent).

    ``heads`` is an optional list of (b, h) pairs; default all.  Returns
    dicts keyed by (b, h): out [len(rows), d], lse [len(rows)].
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, S, H, d = q.shape
    if scale is None:
        scale = default_scale(d)
    pos = natural_positions(lens, zigzag)
    rows = np.asarray(rows, dtype=np.int64)
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    outs, lses = {}, {}
    for (b, h) in heads:
        s = scale * (q[b, rows, h, :] @ k[b, :, h, :].T)
        s = np.where(_visible(pos[rows], pos, causal), s, NEG_INF)
        l_r, p = _softmax_rows(s)
        outs[(b, h)] = p @ v[b, :, h, :]
        lses[(b, h)] = l_r
    return outs, lses


def partial_block(qb, kb, vb, qpos, kpos, causal, scale):
    """One (query shard, KV shard) partial: attention of qb over kb only.

    qb [n, d], kb/vb [m, d].  Returns (O [n, d] normalised, lse [n]); rows with
    no visible key get O = 0 and lse = -inf.
    """
    s = scale * (qb @ kb.T)
    s = np.where(_visible(qpos, kpos, causal), s, NEG_INF)
    lse, p = _softmax_rows(s)
    return p @ vb, lse


def merge_pair(o_a, lse_a, o_b, lse_b):
    """Log-sum-exp merge of two partials over disjoint key sets.

    L = max + log(exp(lse_a - max) + exp(lse_b - max));
    O = exp(lse_a - L) O_a + exp(lse_b - L) O_b.  Both -inf: L = -inf, O = 0.
    """
    lse_a = _as_f64(lse_a)
    lse_b = _as_f64(lse_b)
    m = np.maximum(lse_a, lse_b)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    wa = np.where(finite, np.exp(lse_a - m_safe), 0.0)
    wb = np.where(finite, np.exp(lse_b - m_safe), 0.0)
    tot = wa + wb
    with np.errstate(divide="ignore"):
        L = np.where(finite, m_safe + np.log(np.where(finite, tot, 1.0)), NEG_INF)
    ca = np.where(finite, wa / np.where(finite, tot, 1.0), 0.0)
    cb = np.where(finite, wb / np.where(finite, tot, 1.0), 0.0)
    return ca[..., None] * o_a + cb[..., None] * o_b, L


def merge_partials(partial_out, partial_lse):
    """Merge D partials: partial_out [D, ..., d], partial_lse [D, ...].

    Folds ``merge_pair`` over the leading axis in index order.
    """
    partial_out = _as_f64(partial_out)
    partial_lse = _as_f64(partial_lse)
    o, L = partial_out[0], partial_lse[0]
    for j in range(1, partial_out.shape[0]):
        o, L = merge_pair(o, L, partial_out[j], partial_lse[j])
    return o, L


def kv_visit_order(r: int, D: int, order="ring"):
    """KV shards visited by query shard r, in turn.

    "ring": r, r-1, ..., r+1 (mod D) -- what rank r receives as K/V travel one
    hop per step around a ring; "reverse": r, r+1, ...; a list: an explicit
    permutation used for every r.
    """
    if isinstance(order, (list, tuple, np.ndarray)):
        return [int(j) for j in order]
    if order == "ring":
        return [(r - t) % D for t in range(D)]
    if order == "reverse":
        return [(r + t) % D for t in range(D)]
    raise ValueError(order)


def ring_partials(q, k, v, lens, zigzag=False, causal=False, scale=None):
    """All D x D partials.  Returns (P_out [D, B, S, H, d], P_lse [D, B, H, S]).

    Entry [j] holds, for every query row (of whatever shard), its partial over
    the keys of KV shard j.
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, S, H, d = q.shape
    if scale is None:
        scale = default_scale(d)
    off = shard_offsets(lens)
    pos = natural_positions(lens, zigzag)
    D = len(lens)
    P_out = np.zeros((D, B, S, H, d))
    P_lse = np.zeros((D, B, H, S))
    for r in range(D):
        qs = slice(off[r], off[r + 1])
        for j in range(D):
            ks = slice(off[j], off[j + 1])
            for b in range(B):
                for h in range(H):
                    o, l_ = partial_block(q[b, qs, h], k[b, ks, h], v[b, ks, h],
                                          pos[qs], pos[ks], causal, scale)
                    P_out[j, b, qs, h] = o
                    P_lse[j, b, h, qs] = l_
    return P_out, P_lse


def ring_forward(q, k, v, lens, zigzag=False, causal=False, scale=None, order="ring"):
    """Ring attention: every query shard meets the KV shards in ``order`` and
    folds each partial into a running (O, lse) by the log-sum-exp rule."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, S, H, d = q.shape
    if scale is None:
        scale = default_scale(d)
    off = shard_offsets(lens)
    pos = natural_positions(lens, zigzag)
    D = len(lens)
    out = np.zeros_like(q)
    lse = np.zeros((B, H, S))
    for r in range(D):
        qs = slice(off[r], off[r + 1])
        n = off[r + 1] - off[r]
        for b in range(B):
            for h in range(H):
                o_run = np.zeros((n, d))
                l_run = np.full(n, NEG_INF)
                for j in kv_visit_order(r, D, order):
                    ks = slice(off[j], off[j + 1])
                    o, l_ = partial_block(q[b, qs, h], k[b, ks, h], v[b, ks, h],
                                          pos[qs], pos[ks], causal, scale)
                    o_run, l_run = merge_pair(o_run, l_run, o, l_)
                out[b, qs, h] = o_run
                lse[b, h, qs] = l_run
    return out, lse


def backward(q, k, v, out, lse, dout, lens, zigzag=False, causal=False, scale=None):
    """Gradients (dq, dk, dv) of sum(dout * out) w.r.t. q, k, v (buffer order)."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    out, lse, dout = _as_f64(out), _as_f64(lse), _as_f64(dout)
    B, S, H, d = q.shape
    if scale is None:
        scale = default_scale(d)
    pos = natural_positions(lens, zigzag)
    order = np.argsort(pos, kind="stable")
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    blk = _row_block(S)
    for b in range(B):
        for h in range(H):
            qn, kn, vn = q[b, order, h], k[b, order, h], v[b, order, h]
            on, don = out[b, order, h], dout[b, order, h]
            ln = lse[b, h, order]
            dkn = np.zeros((S, d))
            dvn = np.zeros((S, d))
            for i0 in range(0, S, blk):
                i1 = min(S, i0 + blk)
                s = scale * (qn[i0:i1] @ kn.T)
                if causal:
                    rows = np.arange(i0, i1)[:, None]
                    s = np.where(np.arange(S)[None, :] <= rows, s, NEG_INF)
                p = np.exp(s - ln[i0:i1, None])
                dvn += p.T @ don[i0:i1]
                dp = don[i0:i1] @ vn.T
                delta = np.sum(don[i0:i1] * on[i0:i1], axis=1)
                ds = p * (dp - delta[:, None])
                dq[b, order[i0:i1], h] = scale * (ds @ kn)
                dkn += scale * (ds.T @ qn[i0:i1])
            dk[b, order, h] = dkn
            dv[b, order, h] = dvn
    return dq, dk, dv


def backward_rows(q, k, v, dout, lens, zigzag, causal, rows, scale=None, heads=None):
    """dQ of selected buffer rows, recomputing their out/lse from scratch.

    Returns a dict keyed by (b, h) of dq [len(rows), d].
    """
    q, k, v, dout = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
    B, S, H, d = q.shape
    if scale is None:
        scale = default_scale(d)
    pos = natural_positions(lens, zigzag)
    rows = np.asarray(rows, dtype=np.int64)
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    res = {}
    for (b, h) in heads:
        s = scale * (q[b, rows, h] @ k[b, :, h].T)
        s = np.where(_visible(pos[rows], pos, causal), s, NEG_INF)
        _, p = _softmax_rows(s)
        o = p @ v[b, :, h]
        dp = dout[b, rows, h] @ v[b, :, h].T
        delta = np.sum(dout[b, rows, h] * o, axis=1)
        ds = p * (dp - delta[:, None])
        res[(b, h)] = scale * (ds @ k[b, :, h])
    return res


def row_stats(q, k, v, dout, lens, zigzag=False, causal=False, scale=None, heads=None, workers=1,
              block=256):
    """out, lse and Delta_i = <dO_i, out_i> of every query row of the selected heads.

    The definition again, for long sequences: blocks of query rows in natural
    order, each scored against the keys it can see -- under causal masking a
    block of natural rows [i0, i1) sees only natural keys 0 .. i1-1 (the
    others would enter as exp(-inf) = 0) -- with the keys above a row's own
    position masked inside the block.  Blocks hold independent rows; with
    ``workers`` > 1 they run on a thread pool (numpy releases the interpreter
    lock inside matmul and the elementwise steps).  ``block`` is the number of
    query rows per block.
    Returns three dicts keyed by (b, h): out [S, d], lse [S], delta [S], all in
    buffer order.
    """
    q, k, v, dout = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
    B, S, H, d = q.shape
    if scale is None:
        scale = default_scale(d)
    pos = natural_positions(lens, zigzag)
    order = np.argsort(pos, kind="stable")   # natural position -> buffer row
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    blk = int(block)
    outs, lses, deltas = {}, {}, {}
    for (b, h) in heads:
        qn, kn, vn, don = q[b, order, h], k[b, order, h], v[b, order, h], dout[b, order, h]
        on = np.zeros((S, d))
        ln = np.zeros(S)
        dn = np.zeros(S)

        def block(i0):
            i1 = min(S, i0 + blk)
            n_keys = i1 if causal else S
            s = scale * (qn[i0:i1] @ kn[:n_keys].T)
            if causal:
                rows = np.arange(i0, i1)[:, None]
                s = np.where(np.arange(n_keys)[None, :] <= rows, s, NEG_INF)
            l_blk, p = _softmax_rows(s)
            o = p @ vn[:n_keys]
            on[i0:i1] = o
            ln[i0:i1] = l_blk
            dn[i0:i1] = np.sum(don[i0:i1] * o, axis=1)

        starts = list(range(0, S, blk))
        if workers > 1:
            with ThreadPoolExecutor(workers) as ex:
                list(ex.map(block, starts))
        else:
            for i0 in starts:
                block(i0)
        out_b = np.empty_like(on)
        out_b[order] = on
        lse_b = np.empty_like(ln)
        lse_b[order] = ln
        delta_b = np.empty_like(dn)
        delta_b[order] = dn
        outs[(b, h)], lses[(b, h)], deltas[(b, h)] = out_b, lse_b, delta_b
    return outs, lses, deltas


def backward_cols(q, k, v, dout, lens, zigzag, causal, cols, lse, delta, scale=None, heads=None):
    """dK and dV of selected key columns (buffer rows of k and v).

    Over the queries i that see key j, with P_ij = exp(scale <q_i, k_j> - lse_i):
        dV_j = sum_i P_ij dO_i,
        dK_j = scale sum_i P_ij (<dO_i, v_j> - Delta_i) q_i.
    ``lse`` and ``delta`` are dicts keyed by (b, h) holding every query row's
    lse and Delta (buffer order), e.g. from ``row_stats``.  Returns two dicts
    keyed by (b, h): dk [len(cols), d], dv [len(cols), d].
    """
    q, k, v, dout = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
    B, S, H, d = q.shape
    if scale is None:
        scale = default_scale(d)
    pos = natural_positions(lens, zigzag)
    cols = np.asarray(cols, dtype=np.int64)
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    dks, dvs = {}, {}
    for (b, h) in heads:
        l_h = _as_f64(lse[(b, h)])
        dl_h = _as_f64(delta[(b, h)])
        s = scale * (q[b, :, h] @ k[b, cols, h].T)            # [S queries, n keys]
        vis = _visible(pos, pos[cols], causal)
        p = np.exp(np.where(vis, s - l_h[:, None], NEG_INF))
        dp = dout[b, :, h] @ v[b, cols, h].T
        ds = p * (dp - dl_h[:, None])
        dvs[(b, h)] = p.T @ dout[b, :, h]
        dks[(b, h)] = scale * (ds.T @ q[b, :, h])
    return dks, dvs


def block_grads(qb, kb, vb, dob, lse_b, delta_b, qpos, kpos, causal, scale):
    """One (query shard, KV shard) block's share of the backward.

    qb, dob [n, d] with their rows' full lse_b and Delta_b [n]; kb, vb [m, d].
    Over the visible pairs of the block, with P_ij = exp(s_ij - lse_i):
    dQ_i = scale sum_j dS_ij k_j, dK_j = scale sum_i dS_ij q_i, dV_j = sum_i
    P_ij dO_i.  Summed over every block of a layout these are the gradients of
    ``backward``: each pair (i, j) lies in exactly one block.
    """
    qb, kb, vb, dob = _as_f64(qb), _as_f64(kb), _as_f64(vb), _as_f64(dob)
    lse_b, delta_b = _as_f64(lse_b), _as_f64(delta_b)
    s = scale * (qb @ kb.T)
    vis = _visible(np.asarray(qpos), np.asarray(kpos), causal)
    p = np.exp(np.where(vis, s - lse_b[:, None], NEG_INF))
    dp = dob @ vb.T
    ds = p * (dp - delta_b[:, None])
    return scale * (ds @ kb), scale * (ds.T @ qb), p.T @ dob
