"""Builds a decode layer step from a ``synth`` workload: one paged pool per emulated DCP
shard, filled through the library's ``cp_local_slot`` kernel (slots no request owns stay
NaN), and the shard-local lengths.  Test and benchmark set-up, not part of the library."""
from __future__ import annotations

import torch

import synth
from mla_paged_decode_03_gb300.dcp import build_shard_pool, local_seq_lens
from mla_paged_decode_03_gb300.layer_step import DcpDecodeStep


def step_from_workload(w, device: str = "cuda") -> DcpDecodeStep:
    dev = torch.device(device)
    q = w.q.to(dev)
    kvg = w.kv_global.to(dev)
    bt = w.block_table.to(dev)
    pool_all = synth.poisoned_pool(w.cp * w.num_blocks, w.bs, dev)
    pools, sls = [], []
    for r in range(w.cp):
        pool = pool_all[r * w.num_blocks:(r + 1) * w.num_blocks]
        build_shard_pool(pool, kvg, w.kv_offsets, w.G.tolist(), bt, w.cp, r, w.interleave)
        pools.append(pool)
        sls.append(local_seq_lens(w.G, w.cp, r, w.interleave).to(dev))
    del kvg
    return DcpDecodeStep(q, bt, w.G, pools, sls, w.q_len, w.scale, w.base_e, pool_all=pool_all,
                         causal=w.causal, interleave=w.interleave)
