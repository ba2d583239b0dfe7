"""One rank of a real decode-context-parallel (DCP) group: its shard's partial decode, the
exchange of every rank's (out, lse) over a torch.distributed process group, and the LSE
merge ("vLLM PR #54012" page, section 实现拆解 step 3: the ranks' partial results are
combined through their LSEs, which must share one base; "vLLM PR #48180" page, section
实现拆解: the merge when DCP is on).

Each rank holds its own paged pool (the KV positions it owns under round-robin sharding,
placed there by ``cp_local_slot_scatter``) and calls ``mla_decode`` with its rank; the
partials of all ranks are all-gathered, rank-major, into one [cp, T, H, 512] buffer and
one [cp, T, H] LSE buffer, which ``lse_merge`` reduces.  Every rank ends with the same
merged result.

The exchange is a plain all-gather of dense tensors: no TMA multicast and no library
kernel that reads another GPU's memory.  On one GPU per process the group is NCCL's; the
host logic is tested with gloo ranks on the CPU, where the decode and the merge are
supplied by the caller (the library's kernels need a GPU).
"""
from __future__ import annotations

from typing import Callable, Optional, Tuple

import torch

__all__ = ["DcpGroupDecode"]

Decode = Callable[[int, int], Tuple[torch.Tensor, torch.Tensor]]
Merge = Callable[[torch.Tensor, torch.Tensor], Tuple[torch.Tensor, torch.Tensor]]


class DcpGroupDecode:
    """``decode(rank, world)`` returns this rank's partial (out [T, H, 512], lse [T, H]);
    ``merge(parts [cp, T, H, 512], lses [cp, T, H])`` returns the merged (out, lse).  With
    neither given, the library's ``mla_decode`` arguments must be bound by the caller
    through ``decode`` and the merge is the library's ``lse_merge`` kernel."""

    def __init__(self, decode: Decode, merge: Optional[Merge] = None, group=None,
                 lse_base_e: bool = True):
        import torch.distributed as dist

        self.dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)
        self.decode = decode
        self.lse_base_e = lse_base_e
        self.merge = merge if merge is not None else self._library_merge

    def _library_merge(self, parts: torch.Tensor, lses: torch.Tensor):
        from . import lse_merge

        T, H = lses.shape[1], lses.shape[2]
        out_lse = torch.empty(T, H, dtype=torch.float32, device=lses.device)
        return lse_merge(parts, lses, out_lse=out_lse, lse_base_e=self.lse_base_e)

    def exchange(self, out: torch.Tensor, lse: torch.Tensor):
        """All-gathers every rank's partial, rank-major: returns (parts [cp, T, H, 512],
        lses [cp, T, H]) with this rank's own partial at index ``rank``."""
        out = out.contiguous()
        lse = lse.contiguous()
        parts = torch.empty((self.world,) + tuple(out.shape), dtype=out.dtype, device=out.device)
        lses = torch.empty((self.world,) + tuple(lse.shape), dtype=lse.dtype, device=lse.device)
        self.dist.all_gather(list(parts.unbind(0)), out, group=self.group)
        self.dist.all_gather(list(lses.unbind(0)), lse, group=self.group)
        return parts, lses

    def step(self):
        """This rank's decode, the exchange and the merge: returns the merged (out, lse),
        the same on every rank."""
        out, lse = self.decode(self.rank, self.world)
        parts, lses = self.exchange(out, lse)
        return self.merge(parts, lses)
