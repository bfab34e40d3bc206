"""Seeded synthetic MoBA workloads (shapes and value recipes only).

This module draws random inputs; it holds none of the attention arithmetic.
The shapes follow the pages' settings: block 512 / top-k 3 / 32K context
("Moonshot MoBA paper explained", gsyq.cn/news/227272, sections 1 and 3.1),
block 2048 at long contexts and 4096 at 128K+ ("MOBA mixture of block
attention for server-side long context", hncyxsy.com/news/197418, section 3),
and a 1M-token context (the first page's section 1 speed-up claim).  The pages
name no dataset; these tensors stand in for real activations.

Recipe (all draws from one ``torch.Generator`` per workload, in this order):
q, k, v ~ N(0, 1) (times ``qkv_scale``), then one key-offset vector per
(sequence, block, head) ~ ``offset_std`` * N(0, 1) added to every key of that
block (so the mean-pooled keys differ between blocks and the gate is not
degenerate), then for the "needle" workload: the ids of the needle blocks, the
ids of the needle queries and one direction u ~ N(0, 1)^D shared by all heads,
added to every key of the needle blocks and to every head of the needle
queries; for a "coherent" workload, per (sequence, head, 256-row tile) the
ids of `coherent` distinct past blocks (uniform among the tile's earlier
blocks; all of them when there are fewer) and, added to every query of the
tile, 0.5 times the sum of those blocks' key offsets, so that the tile's rows
agree on their past blocks (the locality real queries often show, which the
other recipes lack).  Values are drawn in fp32 and rounded to bf16 (round to
nearest even).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    seqlens: tuple            # per-sequence token counts
    H: int
    D: int
    block_size: int
    topks: tuple              # top-k values this workload is run with
    seed: int
    qkv_scale: float = 1.0
    offset_std: float = 0.0
    needle_block_frac: float = 0.0
    needle_query_frac: float = 0.0
    varlen: bool = False      # packed [total, H, D] + cu_seqlens instead of [B, S, H, D]
    coherent: int = 0         # > 0: queries of each 256-row tile agree on this many past blocks
    notes: str = ""

    @property
    def total(self) -> int:
        return int(sum(self.seqlens))

    @property
    def B(self) -> int:
        return len(self.seqlens)

    @property
    def S(self) -> int:
        return int(max(self.seqlens))

    def cu_seqlens(self) -> list:
        cu = [0]
        for L in self.seqlens:
            cu.append(cu[-1] + int(L))
        return cu


def _varlen_lengths(seed: int, count: int, lo: int, hi: int) -> tuple:
    g = torch.Generator().manual_seed(seed)
    return tuple(int(x) for x in torch.randint(lo, hi + 1, (count,), generator=g))


WORKLOADS = {
    "tiny": Workload("tiny", (2048,), H=1, D=64, block_size=256, topks=(3,), seed=0,
                     qkv_scale=1.0, offset_std=0.5,
                     notes="B1 H1 S2048 D64 bs256 (8 blocks) top-k 3"),
    "train32k": Workload("train32k", (32768,), H=32, D=128, block_size=512, topks=(3, 64),
                         seed=1, qkv_scale=1.0 / math.sqrt(128.0), offset_std=0.5,
                         notes="B1 H32 S32768 D128 bs512 (64 blocks) top-k 3; top-k 64 = dense"),
    "train8k": Workload("train8k", (8192,), H=32, D=128, block_size=512, topks=(3,),
                        seed=6, qkv_scale=1.0 / math.sqrt(128.0), offset_std=0.5,
                        notes="the 32K training shape cut to 8192 tokens (16 blocks), for "
                              "kernel profiles that must stay small"),
    "long128k": Workload("long128k", (131072,), H=32, D=128, block_size=2048, topks=(3,),
                         seed=2, offset_std=0.5, needle_block_frac=0.05,
                         needle_query_frac=0.01,
                         notes="B1 H32 S131072 D128 bs2048 (64 blocks) top-k 3, needle blocks"),
    "prefill1m": Workload("prefill1m", (1048576,), H=8, D=128, block_size=4096, topks=(3,),
                          seed=3, offset_std=0.5,
                          notes="B1 H8 S1048576 D128 bs4096 (256 blocks) top-k 3"),
    "coherent32k": Workload("coherent32k", (32768,), H=32, D=128, block_size=512, topks=(3,),
                            seed=5, qkv_scale=1.0 / math.sqrt(128.0), offset_std=0.5,
                            coherent=2,
                            notes="the 32K training shape with each 256-row tile's queries "
                                  "agreeing on 2 past blocks"),
    "coherent128k": Workload("coherent128k", (131072,), H=32, D=128, block_size=2048,
                             topks=(3,), seed=7, qkv_scale=1.0 / math.sqrt(128.0),
                             offset_std=0.5, coherent=2,
                             notes="the 128K shape (block 2048) with each 256-row tile's "
                                   "queries agreeing on 2 past blocks"),
    "varlen": Workload("varlen", _varlen_lengths(4, 8, 4096, 65536), H=16, D=128,
                       block_size=512, topks=(1, 2, 3, 4, 8), seed=4, varlen=True,
                       notes="8 sequences, lengths U{4096..65536} (partial tail blocks), "
                             "H16 D128 bs512, top-k in {1,2,3,4,8}"),
}


def custom(seqlens, H, D, block_size, topk, seed=0, qkv_scale=1.0, offset_std=0.5,
           varlen=None, name="custom", coherent=0) -> Workload:
    """A small workload for tests (same recipe, any shape)."""
    seqlens = tuple(int(s) for s in seqlens)
    if varlen is None:
        varlen = len(set(seqlens)) > 1
    return Workload(name, seqlens, H=H, D=D, block_size=block_size, topks=(topk,), seed=seed,
                    qkv_scale=qkv_scale, offset_std=offset_std, varlen=varlen,
                    coherent=coherent)


@dataclass
class Inputs:
    q: torch.Tensor           # [B, S, H, D] or [total, H, D] bf16
    k: torch.Tensor
    v: torch.Tensor
    cu_seqlens: list
    needle_blocks: list = field(default_factory=list)
    needle_queries: list = field(default_factory=list)


def make_inputs(w: Workload, device="cpu") -> Inputs:
    """Draw the workload's q, k, v on ``device`` with a seeded generator."""
    device = torch.device(device)
    g = torch.Generator(device=device).manual_seed(w.seed)
    total, H, D, bs = w.total, w.H, w.D, w.block_size
    shape = (total, H, D)

    def randn(*s):
        return torch.randn(*s, generator=g, device=device, dtype=torch.float32)

    q = randn(*shape).mul_(w.qkv_scale)
    k = randn(*shape).mul_(w.qkv_scale)
    v = randn(*shape).mul_(w.qkv_scale)
    cu = w.cu_seqlens()
    if w.offset_std > 0:
        nblk = [(L + bs - 1) // bs for L in w.seqlens]
        off = randn(sum(nblk), H, D).mul_(w.offset_std)
        # token -> global block id, then add that block's offset
        blk_of_tok = torch.empty(total, dtype=torch.long, device=device)
        base = 0
        for b, L in enumerate(w.seqlens):
            pos = torch.arange(L, device=device) // bs
            blk_of_tok[cu[b]:cu[b + 1]] = pos + base
            base += nblk[b]
        k.add_(off[blk_of_tok])
    needle_blocks, needle_queries = [], []
    if w.needle_block_frac > 0:
        assert w.B == 1
        n = (w.S + bs - 1) // bs
        nb = int(round(w.needle_block_frac * n))
        nq = int(math.ceil(w.needle_query_frac * w.S))
        needle_blocks = sorted(int(x) for x in torch.randperm(n, generator=g, device=device)[:nb])
        needle_queries = sorted(int(x) for x in torch.randperm(w.S, generator=g, device=device)[:nq])
        u = randn(D)
        for c in needle_blocks:
            k[c * bs:(c + 1) * bs] += u
        q[torch.tensor(needle_queries, device=device)] += u
    if w.coherent > 0:
        assert w.offset_std > 0
        tile = 256
        for b, L in enumerate(w.seqlens):
            for t0 in range(0, L, tile):
                c = t0 // bs  # the tile's block (tiles of 256 rows stay in one block when
                #               the block size is a multiple of 256)
                if c == 0:
                    continue
                base_blk = sum(nblk[:b])
                for h in range(H):
                    pick = torch.randperm(c, generator=g, device=device)[:w.coherent]
                    direction = off[base_blk + pick, h, :].sum(0)
                    q[cu[b] + t0: cu[b] + min(t0 + tile, L), h, :] += 0.5 * direction
    q, k, v = (x.to(torch.bfloat16) for x in (q, k, v))
    if not w.varlen:
        q, k, v = (x.view(w.B, w.S, H, D) for x in (q, k, v))
    return Inputs(q, k, v, cu, needle_blocks, needle_queries)


def sample_rows(w: Workload, count: int, seed: int = 1234, needle_queries=()):
    """Seeded (token, head) sample, stratified to always hold the first and last
    token of every sequence, the first and last row of a few blocks, and the
    needle queries."""
    g = torch.Generator().manual_seed(seed)
    cu = w.cu_seqlens()
    bs = w.block_size
    must = set()
    for b in range(w.B):
        s0, L = cu[b], w.seqlens[b]
        must.update({s0, s0 + L - 1})
        n = (L + bs - 1) // bs
        for c in sorted({0, 1, n // 2, n - 1}):
            must.update({s0 + c * bs, s0 + min((c + 1) * bs, L) - 1})
    for t in list(needle_queries)[: count // 8]:
        must.add(int(t))
    toks = sorted(must)
    heads = [int(x) for x in torch.randint(0, w.H, (len(toks),), generator=g)]
    rest = max(0, count - len(toks))
    toks += [int(x) for x in torch.randint(0, w.total, (rest,), generator=g)]
    heads += [int(x) for x in torch.randint(0, w.H, (rest,), generator=g)]
    return toks[:count], heads[:count]


def make_grad(w: Workload, device="cpu", scale: float = 1.0) -> torch.Tensor:
    """Upstream gradient dL/d(out) for the backward pass: N(0, scale^2) in the
    layout of q, from its own generator (seeded with the workload's seed + 7919)
    so that drawing it leaves q, k, v unchanged."""
    device = torch.device(device)
    g = torch.Generator(device=device).manual_seed(w.seed + 7919)
    d = torch.randn(w.total, w.H, w.D, generator=g, device=device, dtype=torch.float32)
    d = d.mul_(scale).to(torch.bfloat16)
    return d if w.varlen else d.view(w.B, w.S, w.H, w.D)
