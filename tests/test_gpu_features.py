"""CUDA path (through the C ABI) against the float64 oracle for the decode variants beyond
the causal, interleave-1 step: non-causal query blocks, round-robin interleave > 1, both
rescale budgets of the tcgen05 kernel, the KV scatter through the slot mapping, and the
refusal of layouts the tcgen05 kernel does not take.

Sources: "vLLM PR #52188 (DSpark + DCP)" page, section 关键源码片段 (the non-causal branch
of _prepare_flattened_decode_metadata; the dcp_span / remainder clamp of the interleave;
cp_local_slot) and section 实现拆解 step 4 (draft KV written through cp_local_slot).
"""
import numpy as np
import pytest
import torch

import mla_paged_decode_03_gb300 as M
import oracle.mla_ref as R
import synth
from mla_paged_decode_03_gb300 import _lib
from step_builder import step_from_workload

import gpu_helpers as H

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(autouse=True)
def _clean():
    M.device_status()
    prev_k = M.set_decode_kernel(M.KERNEL_AUTO)
    prev_b = M.set_rescale_budget(M.BUDGET_AUTO)
    yield
    M.set_decode_kernel(prev_k)
    M.set_rescale_budget(prev_b)


@pytest.fixture(params=["mma", "tc"])
def kernel(request):
    prev = M.set_decode_kernel(M.KERNEL_MMA if request.param == "mma" else M.KERNEL_TC)
    yield request.param
    M.set_decode_kernel(prev)


def _check(w, relative=True, batched=True, with_workspace=True):
    """The layer step of ``w`` against the oracle, shard by shard and merged.  These cases
    (a few keys per shard, query blocks of up to 16 rows) use the derived per-element
    bound of gpu_helpers, 2e-2 + (4 * 2^-8 + 2 (e^delta - 1)) * A: with ~10 keys on a shard
    an output is close to a single |V| (up to ~4 for N(0,1) rows), where the bf16
    roundings of P, of a split partial and of the output alone approach 2e-2."""
    step = step_from_workload(w, DEV)
    step.batched = batched and step.cp > 1
    if not with_workspace:
        step.workspace = torch.empty(0, dtype=torch.uint8, device=DEV)
    out, lse = step.run()
    torch.cuda.synchronize()
    assert M.device_status() == 0
    if relative:
        ro, rl, mo, ml, ra, ma, rd, md = H.oracle_shards(w, with_abs=True)
    else:
        ro, rl, mo, ml = H.oracle_shards(w)
        ra, ma, rd, md = [None] * w.cp, None, [None] * w.cp, None
    if w.cp > 1:
        for r in range(w.cp):
            H.compare(step.partials[r], step.lses[r], ro[r], rl[r], relative,
                      f"{w.name} shard {r}", ra[r], rd[r])
    H.compare(out, lse, mo, ml, relative, f"{w.name} merged", ma, md)
    return step


# ---------------------------------------------------------------------------
# non-causal blocks (every row reads the shard's whole local sequence)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("B_,H_,q_len,lengths,bs,cp", [
    (2, 16, 3, [37, 130], 16, 1),            # tiny shape
    (8, 64, 4, [1100, 64, 2500, 7, 1, 4000, 3333, 129], 64, 2),   # cp2 shape
    (3, 128, 4, [3000, 1234, 77], 64, 8),    # spec shape, reduced
    (2, 128, 16, [900, 40], 64, 4),          # q_len 16
])
@pytest.mark.parametrize("batched", [True, False])
def test_noncausal_blocks(B_, H_, q_len, lengths, bs, cp, batched, kernel):
    w = synth.make_custom(B_, H_, q_len, lengths, bs, cp, base_e=(cp != 2),
                          seed=500 + q_len + cp, causal=False)
    _check(w, batched=batched)


def test_noncausal_rows_equal_single_token_decode():
    # each row of a non-causal block is an ordinary single-token decode of that row
    w = synth.make_custom(2, 64, 4, [700, 2049], 64, 1, seed=510, causal=False)
    step = step_from_workload(w, DEV)
    _, _, mo, ml, _, ma, _, md = H.oracle_shards(w, with_abs=True)
    for i in range(w.q_len):
        qi = step.q[:, i:i + 1].contiguous()
        o1, l1 = M.mla_decode(qi, step.pools[0], step.block_table, step.seq_lens[0], step.gseq,
                              1, 1, 0, step.scale)
        torch.cuda.synchronize()
        rows = [b * w.q_len + i for b in range(w.B)]
        H.compare(o1, l1, mo[rows], ml[rows], True, f"row {i} of a non-causal block, q_len 1",
                  ma[rows], md[rows])
    assert M.device_status() == 0


def test_noncausal_needs_no_global_lengths():
    # a non-causal call reads seq_lens only: causal_seqlens_global may be NULL for cp > 1
    w = synth.make_custom(2, 16, 2, [300, 129], 16, 2, seed=520, causal=False)
    step = step_from_workload(w, DEV)
    ro, rl, _, _, ra, _, rd, _ = H.oracle_shards(w, with_abs=True)
    for r in range(w.cp):
        o, l = M.mla_decode(step.q, step.pools[r], step.block_table, step.seq_lens[r], None,
                            w.q_len, w.cp, r, step.scale, causal=False)
        torch.cuda.synchronize()
        H.compare(o, l, ro[r], rl[r], True, f"non-causal, no global lengths, shard {r}",
                  ra[r], rd[r])
    with pytest.raises(M.MlaError):
        M.mla_decode(step.q, step.pools[0], step.block_table, step.seq_lens[0], None, w.q_len,
                     w.cp, 0, step.scale, causal=True)
    assert M.device_status() == 0


# ---------------------------------------------------------------------------
# interleave > 1 (round-robin segments of I positions)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("il,bs,cp,q_len,lengths", [
    (2, 16, 2, 3, [37, 130, 1]),
    (4, 64, 4, 4, [3000, 129, 66]),
    (16, 64, 8, 2, [2049, 700]),
    (64, 64, 2, 4, [1000, 255]),
    (2, 32, 3, 8, [500, 33]),
])
@pytest.mark.parametrize("batched", [True, False])
def test_interleave(il, bs, cp, q_len, lengths, batched, kernel):
    w = synth.make_custom(len(lengths), 64, q_len, lengths, bs, cp, base_e=True,
                          seed=600 + il + cp, interleave=il)
    _check(w, batched=batched)


@pytest.mark.parametrize("il", [2, 16])
def test_interleave_noncausal(il, kernel):
    w = synth.make_custom(3, 64, 4, [900, 31, 2000], 64, 4, seed=620 + il, interleave=il,
                          causal=False)
    _check(w)


def test_interleave_must_divide_block_size():
    w = synth.make_custom(1, 16, 1, [100], 16, 2, seed=630)
    step = step_from_workload(w, DEV)
    with pytest.raises(M.MlaError) as e:
        M.mla_decode(step.q, step.pools[0], step.block_table, step.seq_lens[0], step.gseq, 1,
                     2, 0, step.scale, interleave=3)
    assert e.value.code == _lib.MLA_ERR_INVALID_ARGUMENT


# ---------------------------------------------------------------------------
# both rescale budgets of the tcgen05 kernel
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("budget", [M.BUDGET_NARROW, M.BUDGET_WIDE])
@pytest.mark.parametrize("name,lengths", [("long", [5000, 4097]), ("cp2", None),
                                          ("spec", [3000, 1234])])
def test_rescale_budgets(name, lengths, budget):
    M.set_rescale_budget(budget)
    w = synth.make_workload(name, lengths=lengths)
    _check(w, relative=True)


@pytest.mark.parametrize("budget", [M.BUDGET_NARROW, M.BUDGET_WIDE])
def test_score_jump_past_the_narrow_float_range(budget):
    """Row 0, head 0 of request 0 sees key B 142 log2 units above its first tile's maximum
    (inside the wide budget: no rescale) and then key C 145 above it (a rescale by
    2^-145, which one fp32 factor cannot hold: B, a quarter of C's weight, would be
    lost).  Both budgets must give the oracle's result."""
    M.set_rescale_budget(budget)
    w = synth.make_custom(2, 16, 2, [3000, 1500], 64, 1, seed=640)
    q0 = w.q[0, 0, 0].double()
    kv = w.kv_global.double()
    s_first = float((w.scale * (kv[:64] @ q0)).max())
    ln2 = float(np.log(2.0))
    for pos, above_log2 in ((100, 142.0), (200, 145.0)):
        c = (s_first + above_log2 * ln2) / w.scale
        kv[pos] = q0 * (c / float(q0 @ q0))
    w.kv_global = kv.to(torch.bfloat16)
    kvb = w.kv_global.double()
    sb = float(w.scale * (kvb[100] @ q0)) - s_first
    sc = float(w.scale * (kvb[200] @ q0)) - s_first
    assert sb / ln2 < 143.5 and 144.5 < sc / ln2 < 146        # the pattern survives bf16
    # no workspace: each request runs whole on one thread-block pair, so the jumps happen
    # inside one online softmax
    _check(w, relative=True, with_workspace=False)


# ---------------------------------------------------------------------------
# cp_local_slot_scatter: new KV rows written through the slot mapping
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("bs,cp,il,N", [(16, 2, 1, 167), (64, 8, 1, 700), (16, 4, 2, 333),
                                        (64, 16, 4, 1500), (32, 1, 1, 99), (8, 3, 2, 50)])
def test_scatter_matches_oracle(bs, cp, il, N):
    g = torch.Generator().manual_seed(bs * 100 + cp * 10 + il)
    B = 3
    vb = (N + bs * cp - 1) // (bs * cp) + 1
    num_blocks = B * vb + 2
    bt = torch.randperm(num_blocks - 1, generator=g)[:B * vb].to(torch.int32).reshape(B, vb)
    pos = torch.randint(-2, N, (B, N), generator=g, dtype=torch.int64)
    for b in range(B):                       # distinct positions per row (one writer per slot)
        perm = torch.randperm(N, generator=g)
        pos[b] = torch.where(pos[b] < 0, pos[b], perm)
    kv_new = torch.randn(B, N, 576, generator=g).to(torch.bfloat16)
    for rank in range(cp):
        pool0 = torch.full((num_blocks, bs, 576), float("nan"), dtype=torch.bfloat16)
        want = R.ref_scatter_kv(H.f64(pool0), pos.numpy(), H.f64(kv_new), bt.numpy(), bs, cp,
                                rank, il)
        pool = pool0.to(DEV)
        slots = torch.empty(B, N, dtype=torch.int64, device=DEV)
        M.cp_local_slot_scatter(pos.to(DEV), kv_new.to(DEV), bt.to(DEV), pool, cp, rank, il,
                                slots=slots)
        got = H.f64(pool)
        assert np.array_equal(np.isnan(got), np.isnan(want))
        fin = ~np.isnan(want)
        assert np.array_equal(got[fin], want[fin])        # copied bit for bit
        assert np.array_equal(slots.cpu().numpy(),
                              R.ref_cp_local_slot(pos.numpy(), bt.numpy(), bs, cp, rank, il))
    assert M.device_status() == 0


def test_scatter_bad_page_is_flagged_not_written():
    bt = torch.tensor([[0, 9]], dtype=torch.int32, device=DEV)    # page 9 is past the cache
    pos = torch.arange(0, 64, dtype=torch.int64, device=DEV).view(1, -1)
    kv_new = torch.ones(1, 64, 576, dtype=torch.bfloat16, device=DEV)
    pool = torch.zeros(4, 16, 576, dtype=torch.bfloat16, device=DEV)
    M.cp_local_slot_scatter(pos, kv_new, bt, pool, 2, 0)
    torch.cuda.synchronize()
    assert M.device_status() & 1
    assert torch.all(pool[0] == 1) and torch.all(pool[1:] == 0)


def test_pools_built_by_scatter_decode_like_the_oracle():
    # the layer step's pools are filled by the scatter kernel (dcp.build_shard_pool)
    w = synth.make_custom(2, 64, 4, [1000, 333], 64, 4, seed=650, interleave=2)
    step = step_from_workload(w, DEV)
    q, rows = H.oracle_workload_rows(w)
    for r in range(w.cp):
        want = R.ref_build_pool(rows, w.block_table.numpy(), w.bs, w.cp, r, w.num_blocks, 2)
        got = H.f64(step.pools[r])
        assert np.array_equal(np.isnan(got), np.isnan(want))
        fin = ~np.isnan(want)
        assert np.array_equal(got[fin], want[fin])


# ---------------------------------------------------------------------------
# layouts the tcgen05 kernel does not take are refused, not run on another kernel
# ---------------------------------------------------------------------------
def test_unsupported_block_size_is_refused():
    w = synth.make_custom(2, 16, 1, [40, 90], 8, 1, seed=660)
    step = step_from_workload(w, DEV)
    with pytest.raises(M.MlaError) as e:
        step.run()
    assert e.value.code == _lib.MLA_ERR_UNSUPPORTED
    M.set_decode_kernel(M.KERNEL_MMA)      # the cross-check kernel takes any block size
    out, lse = step.run()
    torch.cuda.synchronize()
    _, _, mo, ml, _, ma, _, md = H.oracle_shards(w, with_abs=True)
    H.compare(out, lse, mo, ml, True, "block size 8 on the warp-level kernel", ma, md)


@pytest.mark.parametrize("bs", [128, 256])
def test_large_block_sizes(bs):
    w = synth.make_custom(2, 64, 2, [1000, 3000], bs, 2, seed=670 + bs)
    _check(w)
