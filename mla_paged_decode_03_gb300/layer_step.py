"""One decode layer-step over emulated DCP shards on a single GPU.

The KV of every request is split round-robin over ``cp`` shards; each shard has its own
paged pool (built once, outside the step).  A step is: ``mla_decode`` on every shard
(partial out + LSE per shard) followed by ``lse_merge`` of the partials -- the same work a
``cp``-rank DCP group does for one attention layer, with the cross-rank exchange replaced
by the partials landing in one device buffer.  With one shard the step is a single
``mla_decode`` call and no merge.
"""
from __future__ import annotations

from typing import List, Optional

import torch

from . import alloc_workspace, lse_merge, mla_decode
from .dcp import build_shard_pool, local_seq_lens


class DcpDecodeStep:
    def __init__(self, q: torch.Tensor, block_table: torch.Tensor, G: torch.Tensor,
                 pools: List[torch.Tensor], seq_lens: List[torch.Tensor], q_len: int,
                 scale: float, lse_base_e: bool):
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
        self.workspace = alloc_workspace(B, H, q_len, dev)

    @classmethod
    def from_workload(cls, w, device: str = "cuda") -> "DcpDecodeStep":
        """Builds the shard pools of a ``synth`` workload with the library's slot mapping
        (unused slots stay NaN)."""
        import synth  # input generator only: random draws, no method arithmetic

        dev = torch.device(device)
        q = w.q.to(dev)
        kvg = w.kv_global.to(dev)
        bt = w.block_table.to(dev)
        pools, sls = [], []
        for r in range(w.cp):
            pool = synth.poisoned_pool(w.num_blocks, w.bs, dev)
            build_shard_pool(pool, kvg, w.kv_offsets, w.G.tolist(), bt, w.cp, r)
            pools.append(pool)
            sls.append(local_seq_lens(w.G, w.cp, r).to(dev))
        del kvg
        return cls(q, bt, w.G, pools, sls, w.q_len, w.scale, w.base_e)

    def kernel_launches_per_step(self) -> int:
        """Kernels one step launches: per shard the split-KV decode (+ its combine when
        the workspace allows splits), plus the cross-shard merge when cp > 1."""
        from . import workspace_size
        split = 1 if workspace_size(self.B, self.H, self.q_len) > 0 else 0
        return self.cp * (1 + split) + (1 if self.cp > 1 else 0)

    def run(self, stream=None, q: Optional[torch.Tensor] = None):
        q = self.q if q is None else q
        if self.cp == 1:
            mla_decode(q, self.pools[0], self.block_table, self.seq_lens[0], self.gseq,
                       self.q_len, 1, 0, self.scale, out=self.out, lse=self.out_lse,
                       lse_base_e=self.lse_base_e, workspace=self.workspace, stream=stream)
            return self.out, self.out_lse
        for r in range(self.cp):
            mla_decode(q, self.pools[r], self.block_table, self.seq_lens[r], self.gseq,
                       self.q_len, self.cp, r, self.scale, out=self.partials[r],
                       lse=self.lses[r], lse_base_e=self.lse_base_e, workspace=self.workspace,
                       stream=stream)
        lse_merge(self.partials, self.lses, out=self.out, out_lse=self.out_lse,
                  lse_base_e=self.lse_base_e, stream=stream)
        return self.out, self.out_lse
