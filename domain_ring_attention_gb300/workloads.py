"""Seeded synthetic workloads for sharded ring attention.

This module holds the workload recipes only: tensor shapes, sharding shapes,
value distributions and the seeded draws.  It contains none of the attention
arithmetic, none of the shard-layout arithmetic (offsets, zigzag positions)
and is imported by both the CUDA-path tests/bench and the oracle-side tests,
which is the one thing the two sides share.

Recipe (the same for every configuration):
  * q, k, v (and dO for backward) are i.i.d. N(0, std^2) fp32 draws from one
    ``torch.Generator`` seeded with ``seed``, drawn in the order q, k, v, dO,
    then cast to the configuration's dtype (bf16 rounds to nearest-even).
  * The draws fill the buffers directly in buffer ("sharded") order, i.e. shard
    0's tokens, then shard 1's, ...  Because the values are i.i.d. the
    distribution does not depend on the order in which positions are filled,
    so no permutation is needed to build inputs.
  * Layout is BSHD: ``[B, S, H, d]`` contiguous.

The shapes follow the pages' workloads: the ViT image workloads of the
ShardTensor summary (section 4, ViT strong scaling at 1024^2 .. 4096^2 with
16-pixel patches) and the long-sequence 7B causal workload of the TSP summary
(section 4, 16K-128K tokens), as synthetic stand-ins; no dataset is involved.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


def dirichlet_shard_lengths(S: int, D: int, seed: int = 0, multiple: int = 64) -> list[int]:
    """Uneven 'sharding shapes' from a seeded Dirichlet(1) split.

    ShardTensor lets every rank hold a chunk of arbitrary length along the
    sharded axis (ShardTensor summary, section 2, "sharding shapes").  The
    training workload draws those lengths from Dirichlet(1) and rounds them to
    multiples of ``multiple`` tokens:

      p = default_rng(seed).dirichlet(ones(D));  x = p * S / multiple blocks;
      n = max(floor(x), 1);  leftover blocks go one each to the largest
      remainders x - n (ties to the lower index); an overshoot caused by the
      minimum is taken from the largest shard.  sum(n) * multiple == S.
    """
    if S % multiple:
        raise ValueError("S must be a multiple of the rounding unit")
    blocks = S // multiple
    if blocks < D:
        raise ValueError("too few blocks for D shards")
    p = np.random.default_rng(seed).dirichlet(np.ones(D))
    x = p * blocks
    n = np.maximum(np.floor(x).astype(np.int64), 1)
    left = blocks - int(n.sum())
    while left > 0:
        rem = x - n
        i = int(np.argmax(rem))  # argmax returns the lowest index among ties
        n[i] += 1
        left -= 1
    while left < 0:
        i = int(np.argmax(n))
        n[i] -= 1
        left += 1
    return [int(b) * multiple for b in n]


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    d: int
    lens: tuple
    causal: bool
    zigzag: bool
    dtype: str            # "f32" or "bf16"
    std: float = 1.0
    backward: bool = True
    note: str = ""

    @property
    def S(self) -> int:
        return int(sum(self.lens))

    @property
    def D(self) -> int:
        return len(self.lens)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def visible_pairs(self) -> int:
        """Number of (query, key) pairs the method must compute per (b, h)."""
        S = self.S
        return S * (S + 1) // 2 if self.causal else S * S

    def fwd_flops(self) -> int:
        return 4 * self.B * self.H * self.d * self.visible_pairs()

    def bwd_flops(self) -> int:
        return 10 * self.B * self.H * self.d * self.visible_pairs()

    def describe(self) -> dict:
        return {"workload": self.name, "B": self.B, "H": self.H, "head_dim": self.d,
                "S": self.S, "D": self.D, "shard_lens": list(self.lens),
                "causal": self.causal, "zigzag": self.zigzag, "dtype": self.dtype}


def _workloads() -> dict:
    w = {}
    w["tiny_fp32"] = Workload(
        "tiny_fp32", B=1, H=2, d=64, lens=(100, 150, 130, 132), causal=False,
        zigzag=False, dtype="f32", note="S=512, four uneven shards")
    w["vit1024_s4096"] = Workload(
        "vit1024_s4096", B=1, H=16, d=64, lens=(512,) * 8, causal=False,
        zigzag=False, dtype="bf16", std=1.0 / math.sqrt(2.0),
        note="ViT 1024^2 image, patch 16")
    w["vit4096_s65536"] = Workload(
        "vit4096_s65536", B=1, H=16, d=64, lens=(4096,) * 16, causal=False,
        zigzag=False, dtype="bf16", backward=False,
        note="ViT 4096^2 image, patch 16, forward only")
    w["llm7b_causal_s131072"] = Workload(
        "llm7b_causal_s131072", B=1, H=32, d=128, lens=(16384,) * 8, causal=True,
        zigzag=True, dtype="bf16", note="16 zigzag chunks; rank r holds chunks r and 15-r")
    w["train_s32768"] = Workload(
        "train_s32768", B=2, H=32, d=128,
        lens=tuple(dirichlet_shard_lengths(32768, 4, seed=0, multiple=64)),
        causal=True, zigzag=True, dtype="bf16",
        note="Dirichlet(1) sharding shapes rounded to 64, causal zigzag, fwd+bwd")
    return w


WORKLOADS = _workloads()


def make_inputs(wl: Workload, seed: int = 0, device="cpu", with_dout: bool = False,
                heads: int | None = None):
    """Draw q, k, v (and dO) for ``wl`` in buffer order, BSHD, ``wl.dtype``.

    ``heads`` overrides H (used to build reduced-head variants of a workload
    with the same sequence structure).  Returns a tuple of torch tensors on
    ``device``.
    """
    H = wl.H if heads is None else heads
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    shape = (wl.B, wl.S, H, wl.d)
    out = []
    for _ in range(4 if with_dout else 3):
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        if wl.std != 1.0:
            x.mul_(wl.std)
        out.append(x.to(wl.torch_dtype))
    return tuple(out)


def sample_rows(S: int, n: int, seed: int = 1) -> np.ndarray:
    """A seeded, sorted sample of ``n`` distinct buffer rows spread over [0, S).

    The first and last rows are always included so ragged ends are covered.
    """
    n = min(n, S)
    if n <= 2 or S <= 2:
        return np.unique(np.asarray([0, S - 1][:max(n, 1)], dtype=np.int64))
    rng = np.random.default_rng(seed)
    inner = rng.choice(np.arange(1, S - 1), size=min(n - 2, S - 2), replace=False)
    return np.unique(np.concatenate([[0, S - 1], inner]).astype(np.int64))
