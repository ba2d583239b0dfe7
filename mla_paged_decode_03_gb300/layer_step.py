"""One decode layer-step over emulated DCP shards on a single GPU.

The KV of every request is split round-robin over ``cp`` shards; each shard has its own
paged pool (built once, outside the step).  A step is: every shard's partial decode
(partial out + LSE per shard) followed by ``lse_merge`` of the partials -- the same work a
``cp``-rank DCP group does for one attention layer, with the cross-rank exchange replaced
by the partials landing in one device buffer.  The shards run side by side in one
``mla_decode_shards`` launch (their pools are consecutive slices of one cache and their
block-table rows are offset into it), as the ranks of a DCP group run at the same time;
with ``batched = False`` each shard is its own ``mla_decode`` call.  With one shard the
step is a single ``mla_decode`` call and no merge.
"""
from __future__ import annotations

from typing import List, Optional

import torch

from . import _lib, alloc_workspace
from . import _stream


def shard_major_block_table(block_table: torch.Tensor, pool_blocks: List[int]) -> torch.Tensor:
    """Block-table rows of every shard over one cache that holds the shards' pools back to
    back (shard r's pool starts after those of shards 0..r-1): row r*B + b is request b's
    row with its page ids offset into shard r's slice.  An id outside [0, pool_blocks[r])
    becomes -1, so that it stays out of range (flagged, not read from another slice)."""
    rows, base = [], 0
    for nb in pool_blocks:
        ok = (block_table >= 0) & (block_table < nb)
        rows.append(torch.where(ok, block_table + base, torch.full_like(block_table, -1)))
        base += nb
    return torch.cat(rows).contiguous()


class DcpDecodeStep:
    """Buffers and calls of one layer step.  ``pools[r]`` / ``seq_lens[r]`` are shard r's
    paged pool and local lengths, ``G`` the global lengths; ``causal`` False makes every
    query row read its shard's whole sequence; ``interleave`` is the round-robin segment
    length the pools were laid out with."""

    def __init__(self, q: torch.Tensor, block_table: torch.Tensor, G: torch.Tensor,
                 pools: List[torch.Tensor], seq_lens: List[torch.Tensor], q_len: int,
                 scale: float, lse_base_e: bool, pool_all: Optional[torch.Tensor] = None,
                 causal: bool = True, interleave: int = 1):
        self.causal = causal
        self.interleave = interleave
        self.q = q
        self.block_table = block_table
        self.cp = len(pools)
        self.gseq = G.to(device=q.device, dtype=torch.int32)
        self.pools = pools
        self.seq_lens = seq_lens
        self.q_len = q_len
        self.scale = scale
        self.lse_base_e = lse_base_e
        B, _, H, _ = q.shape
        self.B, self.H, self.T = B, H, B * q_len
        dev = q.device
        self.partials = torch.empty(self.cp, self.T, H, 512, dtype=torch.bfloat16, device=dev)
        self.lses = torch.empty(self.cp, self.T, H, dtype=torch.float32, device=dev)
        self.out = torch.empty(self.T, H, 512, dtype=torch.bfloat16, device=dev)
        self.out_lse = torch.empty(self.T, H, dtype=torch.float32, device=dev)
        self.batched = self.cp > 1
        if self.cp > 1:
            # all shards' pages in one cache; shard r's block-table rows point into its slice
            self.pool_all = pool_all if pool_all is not None else torch.cat(pools)
            self.block_table_all = shard_major_block_table(block_table,
                                                           [p.shape[0] for p in pools])
            self.seq_lens_all = torch.cat(seq_lens).contiguous()
        self.workspace = alloc_workspace(self.cp * B, H, q_len, dev)

    def kernel_launches_per_step(self) -> int:
        """Kernels one step launches: per shard the split-KV decode (+ its combine when
        the workspace allows splits), plus the cross-shard merge when cp > 1."""
        from . import workspace_size
        split = 1 if workspace_size(self.B, self.H, self.q_len) > 0 else 0
        calls = 1 if (self.cp == 1 or self.batched) else self.cp
        return calls * (1 + split) + (1 if self.cp > 1 else 0)

    def input_tensors(self) -> List[torch.Tensor]:
        """The per-step device inputs ``run`` reads besides q (block tables, lengths)."""
        if self.cp > 1 and self.batched:
            return [self.block_table_all, self.seq_lens_all, self.gseq]
        return [self.block_table, *self.seq_lens, self.gseq]

    def run(self, stream=None, q: Optional[torch.Tensor] = None):
        """One layer step on ``stream`` (default: the current stream).  The step's buffers
        were checked when they were made, so the library calls go out directly (the C
        entry points still validate every argument)."""
        q = self.q if q is None else q
        L = _lib.load()
        st = _stream(stream)
        ws = self.workspace
        wsb = ws.numel() * ws.element_size()
        base_e = 1 if self.lse_base_e else 0
        scale = float(self.scale)
        causal = 1 if self.causal else 0
        il = int(self.interleave)
        pool0 = self.pools[0]
        if self.cp == 1:
            _lib.check(L.mla_decode(
                q.data_ptr(), pool0.data_ptr(), self.block_table.data_ptr(),
                self.block_table.stride(0), self.seq_lens[0].data_ptr(), self.gseq.data_ptr(),
                self.B, self.H, self.q_len, causal, pool0.shape[1], pool0.shape[0],
                self.block_table.shape[1], 1, 0, il, scale, self.out.data_ptr(),
                self.out_lse.data_ptr(), base_e, ws.data_ptr(), wsb, st))
            return self.out, self.out_lse
        if self.batched:
            bt = self.block_table_all
            _lib.check(L.mla_decode_shards(
                q.data_ptr(), self.pool_all.data_ptr(), bt.data_ptr(), bt.stride(0),
                self.seq_lens_all.data_ptr(), self.gseq.data_ptr(), self.B, self.H, self.q_len,
                causal, pool0.shape[1], self.pool_all.shape[0], bt.shape[1], self.cp, il,
                scale, self.partials.data_ptr(), self.lses.data_ptr(), base_e, ws.data_ptr(),
                wsb, st))
        else:
            bt = self.block_table
            for r in range(self.cp):
                pool = self.pools[r]
                _lib.check(L.mla_decode(
                    q.data_ptr(), pool.data_ptr(), bt.data_ptr(), bt.stride(0),
                    self.seq_lens[r].data_ptr(), self.gseq.data_ptr(), self.B, self.H,
                    self.q_len, causal, pool.shape[1], pool.shape[0], bt.shape[1], self.cp, r,
                    il, scale, self.partials[r].data_ptr(), self.lses[r].data_ptr(), base_e,
                    ws.data_ptr(), wsb, st))
        _lib.check(L.lse_merge(self.partials.data_ptr(), 0, self.lses.data_ptr(), self.cp,
                               self.T, self.H, self.out.data_ptr(), self.out_lse.data_ptr(),
                               base_e, st))
        return self.out, self.out_lse
