"""Host-side helpers for decode context parallelism (DCP) with round-robin KV sharding.

These prepare the inputs that a caller hands to ``mla_decode`` for one shard; they are
not part of the timed decode step.  ``build_shard_pool`` places a request's KV rows into
a shard's paged pool with the library's ``cp_local_slot_scatter`` kernel.
"""
from __future__ import annotations

import torch

from . import cp_local_slot_scatter

__all__ = ["local_seq_lens", "build_shard_pool"]


def local_seq_lens(G: torch.Tensor, cp: int, rank: int, interleave: int = 1) -> torch.Tensor:
    """Shard-local share of global lengths under round-robin sharding in segments of
    ``interleave`` positions ("vLLM PR #52188 (DSpark + DCP)" page, section
    "关键源码片段", _prepare_flattened_decode_metadata): with span = cp*interleave,
    local = G // span * interleave + clamp(G % span - rank*interleave, 0, interleave)."""
    G = G.to(torch.int64)
    span = cp * interleave
    rem = (G % span - rank * interleave).clamp(0, interleave)
    return (G // span * interleave + rem).to(torch.int32)


def build_shard_pool(pool: torch.Tensor, kv_global: torch.Tensor, kv_offsets, G,
                     block_table: torch.Tensor, cp: int, rank: int,
                     interleave: int = 1) -> torch.Tensor:
    """Writes every global KV row this rank owns into ``pool`` [num_blocks, bs, 576] at
    the slot ``cp_local_slot`` gives it, with the ``cp_local_slot_scatter`` kernel, one
    request at a time.  kv_global [sum(G), 576] holds request b's rows at kv_offsets[b];
    block_table [B, max_blocks] int32 is shared by all shards."""
    B = block_table.shape[0]
    G = [int(x) for x in G]
    offs = [int(x) for x in kv_offsets]
    dev = pool.device
    for b in range(B):
        if G[b] == 0:
            continue
        pos = torch.arange(G[b], dtype=torch.int64, device=dev).view(1, -1)
        rows = kv_global[offs[b]:offs[b] + G[b]].view(1, G[b], -1)
        cp_local_slot_scatter(pos, rows, block_table[b:b + 1], pool, cp, rank, interleave)
    return pool
