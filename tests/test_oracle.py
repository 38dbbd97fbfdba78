"""Pins for the oracle: checks against things other than the oracle itself.

* a library attention routine (torch's scaled_dot_product_attention and
  autograd, float64 on the CPU),
* closed forms and hand-worked examples,
* the invariants the pages fix: the sharded, merged result equals unsharded
  attention for any sharding shapes and KV visit order (ShardTensor summary,
  sections 2 and 4); zigzag-causal equals plain causal and balances causal
  work (TSP summary, section 2, attention layer),
* central finite differences for the backward,
* the page's zigzag chunk table (tests/golden/zigzag_8ranks_16chunks.txt).
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import attention as oa
from oracle import bruteforce as ob
from oracle import layout as ol
from domain_ring_attention_gb300.workloads import WORKLOADS, dirichlet_shard_lengths

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def sdpa_f64(qn, kn, vn, causal, scale):
    """torch's attention on natural-order [B,S,H,d] float64 arrays."""
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).permute(0, 2, 1, 3)
    o = torch.nn.functional.scaled_dot_product_attention(
        t(qn), t(kn), t(vn), is_causal=causal, scale=scale)
    return o.permute(0, 2, 1, 3).numpy()


def torch_lse(qn, kn, causal, scale):
    qt = torch.from_numpy(qn).permute(0, 2, 1, 3)
    kt = torch.from_numpy(kn).permute(0, 2, 1, 3)
    s = scale * qt @ kt.transpose(-1, -2)
    if causal:
        S = s.shape[-1]
        s = s.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), -math.inf)
    return torch.logsumexp(s, dim=-1).numpy()


def to_buffer(xn, pos):
    """Place natural-order rows into buffer order: buffer row t holds natural pos[t]."""
    return xn[:, pos]


# ---------------------------------------------------------------- layout

def test_zigzag_chunk_table_matches_page_rule():
    rows = [list(map(int, l.split())) for l in open(os.path.join(GOLDEN, "zigzag_8ranks_16chunks.txt"))
            if l.strip() and not l.startswith("#")]
    lens = [16384] * 8
    pos = ol.natural_positions(lens, zigzag=True)
    c = 8192
    for r, a, b in rows:
        slab = pos[r * 16384:(r + 1) * 16384]
        assert np.array_equal(slab[:c], a * c + np.arange(c))
        assert np.array_equal(slab[c:], b * c + np.arange(c))


@pytest.mark.parametrize("lens", [[2], [4, 4], [6, 2, 10], [64, 12928 // 64 * 2, 384]])
def test_zigzag_positions_are_a_permutation(lens):
    pos = ol.natural_positions(lens, zigzag=True)
    assert np.array_equal(np.sort(pos), np.arange(sum(lens)))
    assert np.array_equal(ol.natural_positions(lens, zigzag=False), np.arange(sum(lens)))


def test_zigzag_rejects_odd_lengths_and_empty_shards():
    with pytest.raises(ValueError):
        ol.natural_positions([3, 4], zigzag=True)
    with pytest.raises(ValueError):
        ol.shard_offsets([4, 0])


@pytest.mark.parametrize("D,c", [(2, 3), (4, 5), (8, 16)])
def test_zigzag_balances_causal_work(D, c):
    """With equal shards every rank owns the same number of visible causal pairs."""
    lens = [2 * c] * D
    pos = ol.natural_positions(lens, zigzag=True)
    owner = ol.shard_of_row(lens)
    work = [int(np.sum(pos[owner == r] + 1)) for r in range(D)]
    assert len(set(work)) == 1
    contiguous = [int(np.sum(np.arange(r * 2 * c, (r + 1) * 2 * c) + 1)) for r in range(D)]
    assert len(set(contiguous)) > 1   # without zigzag the last rank works hardest


def test_dirichlet_shapes_frozen():
    lens = dirichlet_shard_lengths(32768, 4, seed=0, multiple=64)
    assert lens == [12928, 19392, 384, 64]          # frozen at first use
    assert list(WORKLOADS["train_s32768"].lens) == lens
    for seed in range(20):
        for D in (2, 3, 4, 7, 16):
            ls = dirichlet_shard_lengths(32768, D, seed=seed)
            assert sum(ls) == 32768 and all(x % 64 == 0 and x >= 64 for x in ls)


# ---------------------------------------------------------------- forward

@pytest.mark.parametrize("causal", [False, True])
def test_forward_matches_torch_sdpa(causal):
    B, S, H, d = 2, 67, 3, 16
    q, k, v = rnd((B, S, H, d), 1), rnd((B, S, H, d), 2), rnd((B, S, H, d), 3)
    out, lse = oa.forward(q, k, v, [S], zigzag=False, causal=causal)
    ref = sdpa_f64(q, k, v, causal, 1 / math.sqrt(d))
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, torch_lse(q, k, causal, 1 / math.sqrt(d)), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_forward_matches_bruteforce(causal):
    S, d = 11, 5
    q, k, v = rnd((1, S, 1, d), 4), rnd((1, S, 1, d), 5), rnd((1, S, 1, d), 6)
    out, lse = oa.forward(q, k, v, [S], causal=causal, scale=0.37)
    bo, bl = ob.attention(q[0, :, 0].tolist(), k[0, :, 0].tolist(), v[0, :, 0].tolist(),
                          causal=causal, scale=0.37)
    np.testing.assert_allclose(out[0, :, 0], np.array(bo), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], np.array(bl), rtol=1e-12, atol=1e-12)


def test_two_key_worked_example():
    """d = 4 -> scale 1/2; q = e1, k0 = 2 e1, k1 = 0: scores 1 and 0."""
    q = np.zeros((1, 2, 1, 4)); q[0, :, 0, 0] = 1.0
    k = np.zeros((1, 2, 1, 4)); k[0, 0, 0, 0] = 2.0
    v = np.zeros((1, 2, 1, 4)); v[0, 0, 0] = [1, 2, 3, 4]; v[0, 1, 0] = [-1, 0, 5, 0]
    out, lse = oa.forward(q, k, v, [1, 1])
    e = math.e
    assert lse[0, 0, 0] == pytest.approx(math.log(e + 1.0), abs=1e-15)
    want = (e * np.array([1, 2, 3, 4]) + np.array([-1, 0, 5, 0])) / (e + 1)
    np.testing.assert_allclose(out[0, 0, 0], want, rtol=1e-14)
    out_c, lse_c = oa.forward(q, k, v, [2], causal=True)   # row 0 sees only key 0
    np.testing.assert_allclose(out_c[0, 0, 0], [1, 2, 3, 4], rtol=1e-15)
    assert lse_c[0, 0, 0] == pytest.approx(1.0, abs=1e-15)


def test_closed_forms():
    B, S, H, d = 1, 40, 2, 8
    q, v = rnd((B, S, H, d), 7), rnd((B, S, H, d), 8)
    k = np.broadcast_to(rnd((1, 1, H, d), 9), (B, S, H, d)).copy()   # all keys equal
    out, lse = oa.forward(q, k, v, [10, 30])
    np.testing.assert_allclose(out, np.broadcast_to(v.mean(axis=1, keepdims=True), out.shape), atol=1e-13)
    want_lse = np.log(S) + np.einsum("bshd,bhd->bhs", q, k[:, 0]) / math.sqrt(d)
    np.testing.assert_allclose(lse, want_lse, atol=1e-12)
    vc = np.broadcast_to(rnd((1, 1, H, d), 10), (B, S, H, d)).copy()  # all values equal
    out2, _ = oa.forward(q, rnd((B, S, H, d), 11), vc, [S], causal=True)
    np.testing.assert_allclose(out2, vc, atol=1e-13)
    q1, k1, v1 = rnd((1, 1, 1, d), 12), rnd((1, 1, 1, d), 13), rnd((1, 1, 1, d), 14)   # S = 1
    o1, l1 = oa.forward(q1, k1, v1, [1], causal=True)
    np.testing.assert_allclose(o1, v1, rtol=1e-15)
    assert l1[0, 0, 0] == pytest.approx(float(q1.ravel() @ k1.ravel()) / math.sqrt(d), abs=1e-14)


def test_causal_first_natural_row_sees_only_itself_under_zigzag():
    lens = [6, 4, 10]
    S, d = sum(lens), 8
    q, k, v = rnd((1, S, 2, d), 15), rnd((1, S, 2, d), 16), rnd((1, S, 2, d), 17)
    pos = ol.natural_positions(lens, zigzag=True)
    t0 = int(np.where(pos == 0)[0][0])
    out, lse = oa.forward(q, k, v, lens, zigzag=True, causal=True)
    np.testing.assert_allclose(out[0, t0], v[0, t0], rtol=1e-14)
    np.testing.assert_allclose(lse[0, :, t0], np.einsum("hd,hd->h", q[0, t0], k[0, t0]) / math.sqrt(d), atol=1e-14)


def test_zigzag_causal_equals_plain_causal():
    lens = [6, 2, 10, 4]
    S, d = sum(lens), 8
    qn, kn, vn = rnd((2, S, 3, d), 18), rnd((2, S, 3, d), 19), rnd((2, S, 3, d), 20)
    pos = ol.natural_positions(lens, zigzag=True)
    qb, kb, vb = to_buffer(qn, pos), to_buffer(kn, pos), to_buffer(vn, pos)
    out, lse = oa.forward(qb, kb, vb, lens, zigzag=True, causal=True)
    ref = sdpa_f64(qn, kn, vn, True, 1 / math.sqrt(d))
    np.testing.assert_allclose(out, to_buffer(ref, pos), atol=1e-12)
    np.testing.assert_allclose(lse, torch_lse(qn, kn, True, 1 / math.sqrt(d))[:, :, pos], atol=1e-12)


# ---------------------------------------------------------------- ring + merge

RING_CASES = [
    ([5, 1, 7, 3], False, False),
    ([1, 1, 1], False, True),
    ([9, 20, 3, 1, 15], False, True),
    ([6, 2, 10, 4], True, True),
    ([2, 8], True, True),
    ([4, 4, 4, 4, 4, 4, 4, 4], True, True),
    ([12, 2, 6], True, False),
]


@pytest.mark.parametrize("lens,zigzag,causal", RING_CASES)
@pytest.mark.parametrize("order", ["ring", "reverse", "random"])
def test_sharded_merged_equals_unsharded(lens, zigzag, causal, order):
    S, d = sum(lens), 8
    q, k, v = rnd((1, S, 2, d), 21), rnd((1, S, 2, d), 22), rnd((1, S, 2, d), 23)
    if order == "random":
        order = list(np.random.default_rng(len(lens)).permutation(len(lens)))
    out, lse = oa.ring_forward(q, k, v, lens, zigzag, causal, order=order)
    pos = ol.natural_positions(lens, zigzag)
    inv = np.argsort(pos)
    ref = sdpa_f64(q[:, inv], k[:, inv], v[:, inv], causal, 1 / math.sqrt(d))
    np.testing.assert_allclose(out, to_buffer(ref, pos), atol=1e-12)
    full, full_lse = oa.forward(q, k, v, lens, zigzag, causal)
    np.testing.assert_allclose(lse, full_lse, atol=1e-12)


@pytest.mark.parametrize("lens,zigzag,causal", RING_CASES[:4])
def test_partials_then_merge_equals_full(lens, zigzag, causal):
    S, d = sum(lens), 4
    q, k, v = rnd((2, S, 1, d), 24), rnd((2, S, 1, d), 25), rnd((2, S, 1, d), 26)
    P_out, P_lse = oa.ring_partials(q, k, v, lens, zigzag, causal)
    o, L = oa.merge_partials(P_out, P_lse.transpose(0, 1, 3, 2))
    full, full_lse = oa.forward(q, k, v, lens, zigzag, causal)
    np.testing.assert_allclose(o, full, atol=1e-12)
    np.testing.assert_allclose(L.transpose(0, 2, 1), full_lse, atol=1e-12)


def test_merge_identity_and_empty():
    o = rnd((5, 3), 27)
    l_ = rnd((5,), 28)
    m, L = oa.merge_pair(o, l_, np.zeros_like(o), np.full(5, -np.inf))
    np.testing.assert_allclose(m, o, rtol=1e-15)
    np.testing.assert_allclose(L, l_, rtol=1e-15)
    m2, L2 = oa.merge_pair(np.zeros((2, 3)), np.full(2, -np.inf), np.zeros((2, 3)), np.full(2, -np.inf))
    assert np.all(np.isneginf(L2)) and np.all(m2 == 0)


def test_merge_two_halves_closed_form():
    """Two single-key partials: lse = log(e^a + e^b), weights softmax([a, b])."""
    a, b = 0.3, -1.7
    va, vb = np.array([[1.0, -2.0]]), np.array([[4.0, 0.5]])
    m, L = oa.merge_pair(va, np.array([a]), vb, np.array([b]))
    assert L[0] == pytest.approx(math.log(math.exp(a) + math.exp(b)), abs=1e-15)
    wa = math.exp(a) / (math.exp(a) + math.exp(b))
    np.testing.assert_allclose(m[0], wa * va[0] + (1 - wa) * vb[0], rtol=1e-14)


# ---------------------------------------------------------------- backward

def _loss_grad_fd(q, k, v, dout, lens, zigzag, causal, eps=1e-6):
    def loss(qq, kk, vv):
        o, _ = oa.forward(qq, kk, vv, lens, zigzag, causal)
        return float(np.sum(o * dout))
    grads = []
    for which in range(3):
        args = [q.copy(), k.copy(), v.copy()]
        g = np.zeros_like(args[which])
        it = np.nditer(g, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            a = [x.copy() for x in args]
            a[which][idx] += eps
            lp = loss(*a)
            a[which][idx] -= 2 * eps
            lm = loss(*a)
            g[idx] = (lp - lm) / (2 * eps)
        grads.append(g)
    return grads


@pytest.mark.parametrize("lens,zigzag,causal", [([3, 2], False, False), ([4, 2], True, True), ([5], False, True)])
def test_backward_matches_finite_differences(lens, zigzag, causal):
    S, d = sum(lens), 3
    q, k, v, do = (rnd((1, S, 2, d), s) for s in (30, 31, 32, 33))
    out, lse = oa.forward(q, k, v, lens, zigzag, causal)
    dq, dk, dv = oa.backward(q, k, v, out, lse, do, lens, zigzag, causal)
    fq, fk, fv = _loss_grad_fd(q, k, v, do, lens, zigzag, causal)
    np.testing.assert_allclose(dq, fq, atol=1e-8)
    np.testing.assert_allclose(dk, fk, atol=1e-8)
    np.testing.assert_allclose(dv, fv, atol=1e-8)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_torch_autograd(causal):
    B, S, H, d = 1, 37, 2, 8
    q, k, v, do = (rnd((B, S, H, d), s) for s in (34, 35, 36, 37))
    out, lse = oa.forward(q, k, v, [S], causal=causal)
    dq, dk, dv = oa.backward(q, k, v, out, lse, do, [S], causal=causal)
    ts = [torch.from_numpy(x).permute(0, 2, 1, 3).requires_grad_() for x in (q, k, v)]
    o = torch.nn.functional.scaled_dot_product_attention(*ts, is_causal=causal)
    o.backward(torch.from_numpy(do).permute(0, 2, 1, 3))
    for mine, t in zip((dq, dk, dv), ts):
        np.testing.assert_allclose(mine, t.grad.permute(0, 2, 1, 3).numpy(), atol=1e-11)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_single_key_closed_form(causal):
    """One token (S = 1): P = 1 and Delta = dP, so dS = P (dP - Delta) = 0 -- dQ = dK = 0 and dV = dO (the
    textbook backward with a constant softmax).  Catches a Delta or P that is not exactly the forward's."""
    B, H, d = 2, 3, 16
    q, k, v, do = (rnd((B, 1, H, d), s) for s in (61, 62, 63, 64))
    out, lse = oa.forward(q, k, v, [1], causal=causal)
    dq, dk, dv = oa.backward(q, k, v, out, lse, do, [1], causal=causal)
    np.testing.assert_allclose(dv, do, rtol=1e-15)
    scale = np.abs(do).max() * np.abs(v).max() * np.abs(k).max()
    assert np.abs(dq).max() <= 1e-13 * scale and np.abs(dk).max() <= 1e-13 * scale


def test_backward_invariants_under_zigzag():
    lens = [6, 2, 10, 4]
    S, d = sum(lens), 8
    q, k, v, do = (rnd((2, S, 3, d), s) for s in (40, 41, 42, 43))
    out, lse = oa.forward(q, k, v, lens, True, True)
    dq, dk, dv = oa.backward(q, k, v, out, lse, do, lens, True, True)
    # rows of P sum to one -> sum_j dV_j = sum_i dO_i ; rows of dS sum to zero -> sum_j dK_j = 0
    np.testing.assert_allclose(dv.sum(axis=1), do.sum(axis=1), atol=1e-11)
    np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-11)
    # shifting every key by one vector leaves each softmax row, hence dQ, unchanged
    shift = rnd((1, 1, 3, d), 44)
    out2, lse2 = oa.forward(q, k + shift, v, lens, True, True)
    dq2, _, _ = oa.backward(q, k + shift, v, out2, lse2, do, lens, True, True)
    np.testing.assert_allclose(dq2, dq, atol=1e-11)
    # zigzag backward equals natural-order causal backward
    pos = ol.natural_positions(lens, True)
    inv = np.argsort(pos)
    on, ln = oa.forward(q[:, inv], k[:, inv], v[:, inv], [S], False, True)
    gn = oa.backward(q[:, inv], k[:, inv], v[:, inv], on, ln, do[:, inv], [S], False, True)
    for mine, nat in zip((dq, dk, dv), gn):
        np.testing.assert_allclose(mine, to_buffer(nat, pos), atol=1e-11)


# ---------------------------------------------------------------- sampled helpers

def test_sampled_rows_agree_with_full():
    lens = [6, 2, 10, 4]
    S, d = sum(lens), 8
    q, k, v, do = (rnd((2, S, 2, d), s) for s in (50, 51, 52, 53))
    rows = np.array([0, 3, 7, 8, 21])
    out, lse = oa.forward(q, k, v, lens, True, True)
    dq, _, _ = oa.backward(q, k, v, out, lse, do, lens, True, True)
    so, sl = oa.forward_rows(q, k, v, lens, True, True, rows)
    sdq = oa.backward_rows(q, k, v, do, lens, True, True, rows)
    for (b, h), o in so.items():
        np.testing.assert_allclose(o, out[b, rows, h], atol=1e-13)
        np.testing.assert_allclose(sl[(b, h)], lse[b, h, rows], atol=1e-13)
        np.testing.assert_allclose(sdq[(b, h)], dq[b, rows, h], atol=1e-12)


# ---------------------------------------------------------------- planted mistakes

def test_pins_catch_planted_mistakes(monkeypatch):
    """Plant plausible mistakes in the oracle (CPU only) and check a pin fails."""
    B, S, H, d = 1, 9, 1, 4
    q, k, v = rnd((B, S, H, d), 60), rnd((B, S, H, d), 61), rnd((B, S, H, d), 62)
    ref = sdpa_f64(q, k, v, True, 0.5)
    # 1. wrong scale
    monkeypatch.setattr(oa, "default_scale", lambda dd: 1.0 / dd)
    out, _ = oa.forward(q, k, v, [S], causal=True)
    assert not np.allclose(out, ref, atol=1e-6)
    monkeypatch.undo()
    # 2. wrong merge weight sign
    orig = oa.merge_pair
    def bad_merge(oa_, la, ob_, lb):
        o, L = orig(oa_, la, ob_, lb)
        return o, L - 1e-3
    monkeypatch.setattr(oa, "merge_pair", bad_merge)
    _, l_bad = oa.ring_forward(q, k, v, [3, 6], causal=True)
    monkeypatch.undo()
    _, l_ok = oa.forward(q, k, v, [3, 6], causal=True)
    assert not np.allclose(l_bad, l_ok, atol=1e-6)
    # 3. mirrored zigzag chunk (rank r holding 2D-2-r) breaks zigzag == causal
    orig_pos = ol.natural_positions
    def bad_pos(lens, zigzag):
        p = orig_pos(lens, zigzag)
        return p[::-1].copy() if zigzag else p
    monkeypatch.setattr(oa, "natural_positions", bad_pos)
    lens = [4, 6]
    qb = rnd((1, 10, 1, 4), 63)
    out_bad, _ = oa.forward(qb, qb, qb, lens, True, True)
    monkeypatch.undo()
    out_ok, _ = oa.forward(qb, qb, qb, lens, True, True)
    assert not np.allclose(out_bad, out_ok, atol=1e-6)


# ---------------------------------------------------------------- long-sequence helpers

def _natural_autograd(q, k, v, do, lens, zigzag, causal):
    """torch SDPA and autograd in float64 on natural-order copies; results back in buffer order."""
    pos = ol.natural_positions(lens, zigzag)
    inv = np.argsort(pos)
    ts = [torch.from_numpy(np.ascontiguousarray(x[:, inv])).permute(0, 2, 1, 3).requires_grad_()
          for x in (q, k, v)]
    o = torch.nn.functional.scaled_dot_product_attention(*ts, is_causal=causal)
    o.backward(torch.from_numpy(np.ascontiguousarray(do[:, inv])).permute(0, 2, 1, 3))
    back = lambda t: to_buffer(t.detach().permute(0, 2, 1, 3).numpy(), pos)
    lse = torch_lse(np.ascontiguousarray(q[:, inv]), np.ascontiguousarray(k[:, inv]), causal,
                    1 / math.sqrt(q.shape[-1]))
    return back(o), lse[:, :, pos], [back(t.grad) for t in ts]


@pytest.mark.parametrize("lens,zigzag,causal,workers", [
    ([150, 50, 250, 150], True, True, 1), ([150, 50, 250, 150], True, True, 3),
    ([301, 299], False, False, 2), ([600], False, True, 1)])
def test_row_stats_match_torch(lens, zigzag, causal, workers):
    S, d = sum(lens), 8
    q, k, v, do = (rnd((1, S, 2, d), s) for s in (70, 71, 72, 73))
    out_t, lse_t, _ = _natural_autograd(q, k, v, do, lens, zigzag, causal)
    outs, lses, deltas = oa.row_stats(q, k, v, do, lens, zigzag, causal, workers=workers, block=128)
    for (b, h), o in outs.items():
        np.testing.assert_allclose(o, out_t[b, :, h], atol=1e-12)
        np.testing.assert_allclose(lses[(b, h)], lse_t[b, h], atol=1e-12)
        np.testing.assert_allclose(deltas[(b, h)], np.sum(do[b, :, h] * out_t[b, :, h], axis=1), atol=1e-11)


@pytest.mark.parametrize("lens,zigzag,causal", [([150, 50, 250, 150], True, True), ([301, 299], False, False),
                                                ([6, 2, 10, 4], True, True)])
def test_backward_cols_match_torch_autograd(lens, zigzag, causal):
    S, d = sum(lens), 8
    q, k, v, do = (rnd((2, S, 2, d), s) for s in (80, 81, 82, 83))
    _, _, (gq, gk, gv) = _natural_autograd(q, k, v, do, lens, zigzag, causal)
    pos = ol.natural_positions(lens, zigzag)
    # the key of the first natural position (seen by every query), the last one, and a spread
    cols = np.unique(np.concatenate([[int(np.argmin(pos)), int(np.argmax(pos))], np.arange(0, S, 7)]))
    _, lses, deltas = oa.row_stats(q, k, v, do, lens, zigzag, causal, block=64)
    dks, dvs = oa.backward_cols(q, k, v, do, lens, zigzag, causal, cols, lses, deltas)
    for (b, h) in dks:
        np.testing.assert_allclose(dks[(b, h)], gk[b, cols, h], atol=1e-11)
        np.testing.assert_allclose(dvs[(b, h)], gv[b, cols, h], atol=1e-11)
    # and the full oracle backward agrees on those columns
    out, lse = oa.forward(q, k, v, lens, zigzag, causal)
    _, dk, dv = oa.backward(q, k, v, out, lse, do, lens, zigzag, causal)
    np.testing.assert_allclose(dks[(1, 1)], dk[1, cols, 1], atol=1e-11)
    np.testing.assert_allclose(dvs[(1, 1)], dv[1, cols, 1], atol=1e-11)


def test_backward_cols_catch_a_planted_delta_mistake():
    """A Delta taken with the wrong sign (planted here, on the CPU) must fail the autograd pin."""
    lens, S, d = [6, 2, 10, 4], 22, 8
    q, k, v, do = (rnd((1, S, 1, d), s) for s in (90, 91, 92, 93))
    _, _, (_, gk, _) = _natural_autograd(q, k, v, do, lens, True, True)
    _, lses, deltas = oa.row_stats(q, k, v, do, lens, True, True)
    bad = {key: -val for key, val in deltas.items()}
    cols = np.arange(S)
    dks, _ = oa.backward_cols(q, k, v, do, lens, True, True, cols, lses, bad)
    assert not np.allclose(dks[(0, 0)], gk[0, cols, 0], atol=1e-6)


@pytest.mark.parametrize("lens,zigzag,causal", [([6, 2, 10, 4], True, True), ([5, 9, 3], False, False),
                                                ([4, 4], False, True)])
def test_block_grads_sum_to_the_backward(lens, zigzag, causal):
    """Every (query shard, KV shard) block's share, summed over the blocks, gives the full backward
    (itself pinned by autograd and finite differences)."""
    S, d = sum(lens), 8
    q, k, v, do = (rnd((1, S, 2, d), s) for s in (100, 101, 102, 103))
    out, lse = oa.forward(q, k, v, lens, zigzag, causal)
    gq, gk, gv = oa.backward(q, k, v, out, lse, do, lens, zigzag, causal)
    pos = ol.natural_positions(lens, zigzag)
    off = ol.shard_offsets(lens)
    scale = 1 / math.sqrt(d)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for h in range(2):
        delta = np.sum(do[0, :, h] * out[0, :, h], axis=1)
        for r in range(len(lens)):
            qs = slice(off[r], off[r + 1])
            for j in range(len(lens)):
                ks = slice(off[j], off[j + 1])
                a, b, c = oa.block_grads(q[0, qs, h], k[0, ks, h], v[0, ks, h], do[0, qs, h], lse[0, h, qs],
                                         delta[qs], pos[qs], pos[ks], causal, scale)
                dq[0, qs, h] += a
                dk[0, ks, h] += b
                dv[0, ks, h] += c
    np.testing.assert_allclose(dq, gq, atol=1e-12)
    np.testing.assert_allclose(dk, gk, atol=1e-12)
    np.testing.assert_allclose(dv, gv, atol=1e-12)
