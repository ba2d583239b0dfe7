"""Seeded synthetic inputs for paged MLA decode with decode-context-parallel shards.

This module is shared by the oracle side (tests, the CPU baseline) and the CUDA side
(tests, bench).  It draws random numbers and picks the structure of each workload --
context lengths, query/KV values, random page permutations, slot-mapping positions --
and nothing else: it holds none of the method's arithmetic.  In particular it does not
decide which rank owns a position, where a local position lands in a page, or how a
query row is masked; each side does that with its own code.

Workloads (all query/KV values are float32 N(0,1) draws rounded to bf16 with
round-to-nearest-even; head dim 576 = 512 latent + 64 rope; scale 1/sqrt(192)):

  tiny  : B=2,  H=16,  q_len=3, contexts 37 and 130, block_size 16, cp 1, LSE base e,
          plus a slot-mapping case over positions 0..166 with cp_size 2.
  cp2   : B=8,  H=64,  q_len=4, contexts U[1024, 8192], block_size 64, 2 shards,
          LSE base 2, plus slot mapping of each sequence's last 4 positions with the
          last 0..3 of them rejected (encoded as a negative position).
  plain : B=64, H=128, q_len=1, every context 32768, block_size 64, cp 1, base e.
  spec  : B=32, H=128, q_len=4, contexts U[8192, 131072], block_size 64, 8 shards.
  long  : B=4,  H=128, q_len=2, contexts U[262144, 524288], block_size 64, 16 shards,
          1% of KV rows scaled x20, plus slot mapping of 1,048,576 positions, cp_size 8.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch

D_QK = 576          # kv_lora_rank 512 + qk_rope_head_dim 64
D_V = 512           # kv_lora_rank
SCALE = 1.0 / math.sqrt(192.0)   # qk_nope_head_dim 128 + qk_rope_head_dim 64

CONFIGS = {
    "tiny": dict(B=2, H=16, q_len=3, ctx=(37, 130), bs=16, cp=1, base_e=True, seed=0,
                 outlier_frac=0.0),
    "cp2": dict(B=8, H=64, q_len=4, ctx=("uniform", 1024, 8192), bs=64, cp=2, base_e=False,
                seed=1, outlier_frac=0.0),
    "plain": dict(B=64, H=128, q_len=1, ctx=("fixed", 32768), bs=64, cp=1, base_e=True,
                  seed=2, outlier_frac=0.0),
    "spec": dict(B=32, H=128, q_len=4, ctx=("uniform", 8192, 131072), bs=64, cp=8,
                 base_e=True, seed=3, outlier_frac=0.0),
    "long": dict(B=4, H=128, q_len=2, ctx=("uniform", 262144, 524288), bs=64, cp=16,
                 base_e=True, seed=4, outlier_frac=0.01),
}
ORDER = ["tiny", "cp2", "plain", "spec", "long"]


@dataclasses.dataclass
class SlotCase:
    """Inputs of one slot-mapping case: positions [Bs, N] (negative = rejected)."""
    positions: torch.Tensor      # int64 [Bs, N]
    block_table: torch.Tensor    # int32 [Bs, max_blocks]
    block_size: int
    cp_size: int
    interleave: int


@dataclasses.dataclass
class Workload:
    name: str
    B: int
    H: int
    q_len: int
    bs: int
    cp: int
    base_e: bool
    scale: float
    G: torch.Tensor              # int64 [B] global context length per request
    q: torch.Tensor              # bf16 [B, q_len, H, 576]
    kv_global: torch.Tensor      # bf16 [sum(G), 576], request b's rows at kv_offsets[b]
    kv_offsets: torch.Tensor     # int64 [B+1]
    block_table: torch.Tensor    # int32 [B, max_blocks], shared by every shard's pool
    num_blocks: int              # pages in each shard's pool (the last one is a spare)
    slot_cases: List[SlotCase]
    interleave: int = 1          # round-robin segment length of the KV sharding
    causal: bool = True          # False: every query row sees the whole context

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    def rows_of(self, b: int) -> torch.Tensor:
        o = self.kv_offsets
        return self.kv_global[int(o[b]):int(o[b + 1])]


def _draw_lengths(spec, B, gen):
    kind = spec[0] if isinstance(spec[0], str) else "list"
    if kind == "list":
        return torch.tensor(spec, dtype=torch.int64)
    if kind == "fixed":
        return torch.full((B,), int(spec[1]), dtype=torch.int64)
    lo, hi = int(spec[1]), int(spec[2])
    return torch.randint(lo, hi + 1, (B,), generator=gen, dtype=torch.int64)


def _randn_bf16(shape, gen, device):
    return torch.randn(shape, generator=gen, dtype=torch.float32, device=device).to(torch.bfloat16)


def make_workload(name: str, device: str = "cpu", lengths: Optional[List[int]] = None,
                  B: Optional[int] = None, draw_values: bool = True) -> Workload:
    """Draw one workload.  ``lengths``/``B`` shrink a workload for quick tests while
    keeping its structure (head count, q_len, block size, shard count, LSE base).  With
    ``draw_values`` False the query and KV values are not drawn (empty tensors); the
    lengths, block table and slot-mapping cases are the same as with them."""
    c = dict(CONFIGS[name])
    if B is not None:
        c["B"] = B
    seed = c["seed"]
    hgen = torch.Generator().manual_seed(seed)
    if lengths is not None:
        G = torch.tensor(lengths, dtype=torch.int64)
        c["B"] = len(lengths)
    else:
        G = _draw_lengths(c["ctx"], c["B"], hgen)
        if len(G) != c["B"]:
            c["B"] = len(G)
    Bn, H, q_len, bs, cp = c["B"], c["H"], c["q_len"], c["bs"], c["cp"]

    total = int(G.sum())
    if draw_values:
        dgen = torch.Generator(device=device).manual_seed(seed + 1000)
        q = _randn_bf16((Bn, q_len, H, D_QK), dgen, device)
        kvf = torch.randn((total, D_QK), generator=dgen, dtype=torch.float32, device=device)
        if c["outlier_frac"] > 0:
            n_out = max(1, int(round(total * c["outlier_frac"])))
            idx = torch.randint(0, total, (n_out,), generator=dgen, device=device)
            kvf[idx] *= 20.0
        kv_global = kvf.to(torch.bfloat16)
        del kvf
    else:
        q = torch.empty((0,), dtype=torch.bfloat16, device=device)
        kv_global = torch.empty((0, D_QK), dtype=torch.bfloat16, device=device)
    offsets = torch.zeros(Bn + 1, dtype=torch.int64)
    offsets[1:] = torch.cumsum(G, 0)

    # Page budget per request and per shard: enough pages for ceil(G/span) segments of
    # `interleave` tokens, which bounds the share of any shard.  One spare column per row
    # points at the spare page so that reads past a request's pages would be visible.
    il = int(c.get("interleave", 1))
    span = cp * il
    per_shard_tokens = (G + span - 1) // span * il
    pages = (per_shard_tokens + bs - 1) // bs
    total_pages = int(pages.sum())
    num_blocks = total_pages + 1
    spare = num_blocks - 1
    max_blocks = int(pages.max()) + 1
    perm = torch.randperm(total_pages, generator=hgen).to(torch.int32)
    bt = torch.full((Bn, max_blocks), spare, dtype=torch.int32)
    o = 0
    for b in range(Bn):
        n = int(pages[b])
        bt[b, :n] = perm[o:o + n]
        o += n

    slot_cases: List[SlotCase] = []
    if name == "tiny":
        # one sequence over positions 0..166 under cp_size 2 (block table >= 6 virtual
        # blocks), and each request's own positions 0..G-1 under cp_size 2.
        sbt = torch.randperm(64, generator=hgen)[:8].to(torch.int32).reshape(1, 8)
        slot_cases.append(SlotCase(torch.arange(167, dtype=torch.int64).reshape(1, 167), sbt,
                                   bs, 2, 1))
        Nmax = int(G.max())
        pos = torch.full((Bn, Nmax), -1, dtype=torch.int64)
        for b in range(Bn):
            pos[b, :int(G[b])] = torch.arange(int(G[b]))
        vb = (Nmax + 2 * bs - 1) // (2 * bs)
        sbt2 = torch.randperm(4 * vb * Bn, generator=hgen)[:Bn * vb].to(torch.int32).reshape(Bn, vb)
        slot_cases.append(SlotCase(pos, sbt2, bs, 2, 1))
    elif name == "cp2":
        # draft block of the last 4 positions; the last r ~ U{0..3} are rejected.
        pos = G.reshape(-1, 1) - 4 + torch.arange(4, dtype=torch.int64).reshape(1, 4)
        r = torch.randint(0, 4, (Bn,), generator=hgen)
        for b in range(Bn):
            if int(r[b]) > 0:
                pos[b, 4 - int(r[b]):] = -1
        slot_cases.append(SlotCase(pos, bt.clone(), bs, cp, 1))
    elif name == "long":
        # 1,048,576 positions in total: the last 262,144 positions of each sequence.
        Bs = Bn
        N = 1048576 // Bs
        pos = G.reshape(-1, 1) - N + torch.arange(N, dtype=torch.int64).reshape(1, N)
        scp = 8
        vb = int((int(G.max()) + bs * scp - 1) // (bs * scp))
        sbt = torch.randperm(Bs * vb * 2, generator=hgen)[:Bs * vb].to(torch.int32).reshape(Bs, vb)
        slot_cases.append(SlotCase(pos, sbt, bs, scp, 1))

    return Workload(name=name, B=Bn, H=H, q_len=q_len, bs=bs, cp=cp, base_e=c["base_e"],
                    scale=SCALE, G=G, q=q, kv_global=kv_global, kv_offsets=offsets,
                    block_table=bt, num_blocks=num_blocks, slot_cases=slot_cases,
                    interleave=il, causal=bool(c.get("causal", True)))


def make_custom(B: int, H: int, q_len: int, lengths, bs: int, cp: int, base_e: bool = True,
                seed: int = 0, outlier_frac: float = 0.0, device: str = "cpu",
                spare_columns: int = 1, interleave: int = 1, causal: bool = True) -> Workload:
    """An ad-hoc workload with the same drawing rules (edge-case tests); ``interleave``
    sizes the pages for round-robin segments of that length, ``causal`` False marks the
    query blocks non-causal (every row sees the whole context)."""
    name = f"custom_{seed}"
    CONFIGS[name] = dict(B=B, H=H, q_len=q_len, ctx=tuple(lengths), bs=bs, cp=cp,
                         base_e=base_e, seed=seed, outlier_frac=outlier_frac,
                         interleave=interleave, causal=causal)
    try:
        w = make_workload(name, device=device, lengths=list(lengths))
    finally:
        del CONFIGS[name]
    if spare_columns != 1:
        bt = w.block_table
        extra = torch.full((bt.shape[0], spare_columns), w.num_blocks - 1, dtype=torch.int32)
        w.block_table = torch.cat([bt[:, :-1], extra], 1) if spare_columns > 0 else bt[:, :-1]
    w.name = name
    return w


def poisoned_pool(num_blocks: int, bs: int, device: str = "cpu") -> torch.Tensor:
    """A shard pool [num_blocks, bs, 576] bf16 filled with NaN; every slot that a
    request does not own stays NaN, so any read outside the visible set shows up."""
    return torch.full((num_blocks, bs, D_QK), float("nan"), dtype=torch.bfloat16, device=device)
