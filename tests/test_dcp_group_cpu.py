"""A real DCP group on CPU: gloo ranks, each with its own shard pool.

Each rank builds the pool of the KV positions it owns (the oracle's slot mapping, with
interleave), computes its partial with the oracle's shard decode, and the library's
DcpGroupDecode exchanges the partials over the process group and merges them (here with
the oracle's merge: the library's merge kernel needs a GPU).  Every rank's merged result
must equal unsharded attention ("vLLM PR #54012" page, section 实现拆解 step 3), and the
gathered partials must sit in rank order, for 2 and 3 ranks.
"""
import math
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _inputs(seed, B, H, q_len, G, bs, cp, il):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, q_len, H, 576, generator=g).to(torch.bfloat16).double().numpy()
    rows = [torch.randn(int(n), 576, generator=g).to(torch.bfloat16).double().numpy() for n in G]
    ppr = max(((n + cp * il - 1) // (cp * il) * il + bs - 1) // bs for n in G)
    perm = torch.randperm(B * ppr, generator=g).numpy().reshape(B, ppr)
    bt = np.concatenate([perm, np.full((B, 1), B * ppr)], 1)
    return q, rows, bt, B * ppr + 1


def _worker(rank, world, port, il, causal, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle.mla_ref as R
    from mla_paged_decode_03_gb300.dcp_group import DcpGroupDecode

    B, H, q_len, G, bs = 2, 4, 3, (70, 131), 8
    scale = 1.0 / math.sqrt(192.0)
    q, rows, bt, nb = _inputs(7, B, H, q_len, G, bs, world, il)
    Ga = np.array(G)

    def decode(r, cp):
        pool = R.ref_build_pool(rows, bt, bs, cp, r, nb, il)      # this rank's own pool only
        sl = R.ref_local_len(Ga, cp, r, il)
        o, l = R.ref_mla_decode(q, pool, bt, sl, Ga, q_len, cp, r, scale, True, interleave=il,
                                causal=causal)
        return torch.from_numpy(o).float(), torch.from_numpy(l).float()

    def merge(parts, lses):
        o, l = R.ref_lse_merge(parts.double().numpy(), lses.double().numpy(), True)
        return torch.from_numpy(o), torch.from_numpy(l)

    step = DcpGroupDecode(decode, merge)
    assert (step.rank, step.world) == (rank, world)
    # the exchange puts rank k's partial at index k on every rank
    parts, lses = step.exchange(*decode(rank, world))
    for k in range(world):
        ok, lk = decode(k, world)
        assert torch.equal(parts[k], ok) and torch.equal(lses[k], lk), (rank, k)
    mo, ml = step.step()
    go, gl = R.ref_attention_global(q, rows, Ga, q_len, scale, causal=causal)
    # the partials were exchanged as float32: a float32 rounding of each, then the merge
    err = float(np.abs(mo.numpy() - go).max())
    lerr = float(np.abs(ml.numpy() - gl).max())
    out[rank] = (err, lerr)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world,il,causal", [(2, 1, True), (3, 2, True), (2, 4, False)])
def test_dcp_group_exchange_and_merge(world, il, causal):
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, il, causal, out))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    for r in range(world):
        err, lerr = out[r]
        assert err < 1e-5 and lerr < 1e-5, (r, err, lerr)
