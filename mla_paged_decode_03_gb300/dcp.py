"""Host-side helpers for decode context parallelism (DCP) with round-robin KV sharding.

These prepare the inputs that a caller hands to ``mla_decode`` for one shard; they are
not part of the timed decode step.  ``build_shard_pool`` places a request's KV rows into
a shard's paged pool with the library's ``cp_local_slot`` kernel.
"""
from __future__ import annotations

import torch

from . import cp_local_slot

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
    the slot ``cp_local_slot`` gives it.  kv_global [sum(G), 576] holds request b's rows
    at kv_offsets[b]; block_table [B, max_blocks] int32 is shared by all shards."""
    B = block_table.shape[0]
    G = [int(x) for x in G]
    offs = [int(x) for x in kv_offsets]
    Gmax = max(G) if G else 0
    if Gmax == 0:
        return pool
    dev = pool.device
    pos = torch.arange(Gmax, dtype=torch.int64, device=dev).repeat(B, 1)
    lens = torch.tensor(G, dtype=torch.int64, device=dev).view(B, 1)
    pos = torch.where(pos < lens, pos, torch.full_like(pos, -1))
    slots = cp_local_slot(pos, block_table, pool.shape[1], cp, rank, interleave)
    flat = pool.view(-1, pool.shape[2])
    src_index = (torch.tensor(offs[:B], dtype=torch.int64, device=dev).view(B, 1)
                 + torch.arange(Gmax, dtype=torch.int64, device=dev).view(1, Gmax))
    own = slots >= 0
    flat.index_copy_(0, slots[own], kv_global.index_select(0, src_index[own]))
    return pool
