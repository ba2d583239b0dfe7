"""CUDA path (through the C ABI) against the float64 oracle, element by element.

Slot mapping must be bit-exact; decode outputs and merged outputs must be within the
tolerances stated in gpu_helpers.  Pools are filled with NaN wherever no KV row lives,
so a read of an unreferenced page or of a slot past a request's length shows up as a
non-finite output.
"""
import numpy as np
import pytest
import torch

import mla_paged_decode_03_gb300 as M
import oracle.mla_ref as R
import synth
from mla_paged_decode_03_gb300.dcp import build_shard_pool, local_seq_lens
from step_builder import step_from_workload

import gpu_helpers as H

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _clean_status():
    M.device_status()
    yield
    M.set_decode_kernel(M.KERNEL_AUTO)


@pytest.fixture(autouse=True)
def _status_clear():
    """Every test starts with a clean device status word."""
    M.device_status()
    yield


@pytest.fixture(params=["mma", "tc"])
def kernel(request):
    """Runs a decode test once per decode kernel (warp-level mma.sync, tcgen05)."""
    prev = M.set_decode_kernel(M.KERNEL_MMA if request.param == "mma" else M.KERNEL_TC)
    yield request.param
    M.set_decode_kernel(prev)


# ---------------------------------------------------------------------------
# cp_local_slot
# ---------------------------------------------------------------------------
def _slot_case_check(case):
    pos = case.positions
    bt = case.block_table
    for rank in range(case.cp_size):
        want = R.ref_cp_local_slot(pos.numpy(), bt.numpy(), case.block_size, case.cp_size, rank,
                                   case.interleave)
        got = M.cp_local_slot(pos.to(DEV), bt.to(DEV), case.block_size, case.cp_size, rank,
                              case.interleave).cpu().numpy()
        assert np.array_equal(got, want), (rank, np.argwhere(got != want)[:5])
    assert M.device_status() == 0


@pytest.mark.parametrize("name", ["tiny", "cp2", "long"])
def test_cp_local_slot_workloads(name):
    # every position of every case, every rank, bit-exact (the long workload's case is
    # 1,048,576 positions with cp_size 8: the oracle loops over them once per rank)
    w = synth.make_workload(name, draw_values=False)
    assert w.slot_cases
    for case in w.slot_cases:
        _slot_case_check(case)


@pytest.mark.parametrize("bs,cp,il,N", [(16, 2, 1, 167), (64, 8, 1, 1000), (16, 4, 2, 333),
                                        (64, 16, 4, 2048), (32, 1, 1, 99), (8, 3, 2, 50),
                                        (64, 2, 64, 640)])
def test_cp_local_slot_shapes(bs, cp, il, N):
    g = torch.Generator().manual_seed(bs * 1000 + cp * 10 + il)
    B = 3
    vb = (N + bs * cp - 1) // (bs * cp) + 1
    bt = torch.randperm(B * vb * 3, generator=g)[:B * vb].to(torch.int32).reshape(B, vb)
    pos = torch.randint(-3, N, (B, N), generator=g, dtype=torch.int64)
    _slot_case_check(synth.SlotCase(pos, bt, bs, cp, il))


def test_cp_local_slot_padded_table_stride():
    bs, cp = 16, 2
    bt_full = torch.randperm(64, generator=torch.Generator().manual_seed(1))[:24].to(
        torch.int32).reshape(2, 12)
    bt = bt_full[:, :5]                                  # row stride 12, 5 valid columns
    pos = torch.arange(0, 160, dtype=torch.int64).repeat(2, 1)
    for rank in range(cp):
        want = R.ref_cp_local_slot(pos.numpy(), bt.numpy(), bs, cp, rank, 1)
        got = M.cp_local_slot(pos.to(DEV), bt_full.to(DEV)[:, :5], bs, cp, rank).cpu().numpy()
        assert np.array_equal(got, want)


def test_cp_local_slot_out_of_table_flags_status():
    bt = torch.tensor([[3, 5]], dtype=torch.int32, device=DEV)
    pos = torch.tensor([[0, 1, 62, 63, 64, 65, 1000, -2]], dtype=torch.int64, device=DEV)
    got = M.cp_local_slot(pos, bt, 16, 2, 0).cpu().numpy()[0]
    assert list(got[4:]) == [-1, -1, -1, -1]              # virtual block 2+ is past the table
    assert list(got[:4]) == [48, -1, 5 * 16 + 15, -1]     # 63 is rank 1's
    assert M.device_status() & 4


# ---------------------------------------------------------------------------
# lse_merge
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("n,fp32,base_e", [(1, False, True), (2, False, False), (8, False, True),
                                           (16, True, True), (3, True, False), (40, False, True)])
def test_lse_merge_parity(n, fp32, base_e):
    g = torch.Generator().manual_seed(n * 7 + fp32)
    T, Hh = 13, 24
    parts = torch.randn(n, T, Hh, 512, generator=g)
    parts = parts.to(torch.float32 if fp32 else torch.bfloat16)
    lses = torch.randn(n, T, Hh, generator=g) * 5 + 10
    empty = torch.rand(n, T, Hh, generator=g) < 0.3
    lses[empty] = float("-inf")
    lses[:, 0, 0] = float("-inf")                         # a row with no shard at all
    wo, wl = R.ref_lse_merge(H.f64(parts), H.f64(lses), base_e)
    out, ol = M.lse_merge(parts.to(DEV), lses.to(DEV), out_lse=torch.empty(T, Hh, device=DEV),
                          lse_base_e=base_e)
    H.compare(out, ol, wo, wl, what=f"merge n={n}")
    assert torch.all(out[0, 0] == 0)


@pytest.mark.parametrize("n,T,Hh", [(12, 7, 5), (33, 3, 3), (64, 1, 1), (9, 1, 3)])
def test_lse_merge_few_rows_many_shards(n, T, Hh):
    # few rows of many shards take several warps per row (each a strided subset of the
    # shards, summed through shared memory): odd row counts, fewer rows than a block holds
    g = torch.Generator().manual_seed(n * 13 + T)
    parts = torch.randn(n, T, Hh, 512, generator=g).to(torch.bfloat16)
    lses = torch.randn(n, T, Hh, generator=g) * 5 + 10
    lses[torch.rand(n, T, Hh, generator=g) < 0.3] = float("-inf")
    lses[:, -1, -1] = float("-inf")                       # a row with no shard at all
    parts[:, -1, -1] = float("nan")                       # never read: every weight is 0
    wo, wl = R.ref_lse_merge(H.f64(parts), H.f64(lses), True)
    out, ol = M.lse_merge(parts.to(DEV), lses.to(DEV), out_lse=torch.empty(T, Hh, device=DEV))
    H.compare(out, ol, wo, wl, what=f"merge n={n} rows={T * Hh}")
    assert torch.all(out[-1, -1] == 0)


def test_lse_merge_skips_nan_partials_of_empty_shards():
    parts = torch.randn(2, 4, 8, 512).to(torch.bfloat16)
    parts[1] = float("nan")
    lses = torch.randn(2, 4, 8)
    lses[1] = float("-inf")
    out, _ = M.lse_merge(parts.to(DEV), lses.to(DEV))
    assert torch.allclose(out.float().cpu(), parts[0].float(), atol=0, rtol=0)


# ---------------------------------------------------------------------------
# mla_decode: whole workloads at sizes the oracle finishes in seconds
# ---------------------------------------------------------------------------
def _gpu_shards(w, with_workspace=True, batched=True):
    step = step_from_workload(w, DEV)
    step.batched = batched and step.cp > 1
    if not with_workspace:
        step.workspace = torch.empty(0, dtype=torch.uint8, device=DEV)
    return step


def _check_workload(w, relative=False, with_workspace=True, batched=True):
    step = _gpu_shards(w, with_workspace, batched)
    out, lse = step.run()
    torch.cuda.synchronize()
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
    assert M.device_status() == 0


def test_decode_tiny_full(kernel):
    _check_workload(synth.make_workload("tiny"))


def test_decode_cp2_full(kernel):
    _check_workload(synth.make_workload("cp2"))


@pytest.mark.parametrize("name,lengths", [
    ("plain", [1000, 777, 2049]),
    ("spec", [3000, 1234]),
    ("long", [5000, 4097]),
])
def test_decode_reduced_workloads(name, lengths, kernel):
    _check_workload(synth.make_workload(name, lengths=lengths), relative=(name == "long"))


@pytest.mark.parametrize("with_workspace", [True, False])
@pytest.mark.parametrize("name,lengths", [("cp2", None), ("spec", [3000, 1234, 77])])
def test_decode_shard_by_shard_calls(name, lengths, with_workspace, kernel):
    # the per-shard entry point (one mla_decode call per rank) against the oracle, as the
    # layer step runs it with batched = False
    _check_workload(synth.make_workload(name, lengths=lengths), with_workspace=with_workspace,
                    batched=False)


def test_decode_shards_matches_per_shard_calls(kernel):
    # one launch over all shards and one call per shard compute the same partials
    w = synth.make_custom(3, 64, 4, [900, 65, 2100], 64, 4, base_e=False, seed=77)
    a = _gpu_shards(w, batched=True)
    a.run()
    b = _gpu_shards(w, batched=False)
    b.run()
    torch.cuda.synchronize()
    assert M.device_status() == 0
    ro, rl, _, _ = H.oracle_shards(w)
    for r in range(w.cp):
        H.compare(a.partials[r], a.lses[r], ro[r], rl[r], False, f"batched shard {r}")
        H.compare(b.partials[r], b.lses[r], ro[r], rl[r], False, f"per-shard call {r}")
    assert (a.partials.float() - b.partials.float()).abs().max().item() <= 2e-2
    assert (a.lses - b.lses).abs().max().item() <= 1e-3


def test_decode_shards_python_wrapper_and_one_shard(kernel):
    # the wrapper's own allocations give the layer step's partials bit for bit (the kernel
    # is deterministic), and one shard through mla_decode_shards is mla_decode
    w = synth.make_custom(3, 64, 2, [700, 64, 1300], 64, 2, base_e=True, seed=21)
    step = _gpu_shards(w)
    step.run()
    out, lse = M.mla_decode_shards(step.q, step.pool_all, step.block_table_all,
                                   step.seq_lens_all, step.gseq, step.q_len, step.cp,
                                   step.scale, lse_base_e=step.lse_base_e)
    torch.cuda.synchronize()
    assert out.shape == step.partials.shape and lse.shape == step.lses.shape
    assert torch.equal(out, step.partials) and torch.equal(lse, step.lses)
    w1 = synth.make_custom(2, 128, 1, [900, 2049], 64, 1, base_e=True, seed=22)
    s1 = _gpu_shards(w1)
    o1, l1 = s1.run()
    o2, l2 = M.mla_decode_shards(s1.q, s1.pools[0], s1.block_table, s1.seq_lens[0], s1.gseq,
                                 s1.q_len, 1, s1.scale, lse_base_e=True)
    torch.cuda.synchronize()
    assert torch.equal(o2[0], o1) and torch.equal(l2[0], l1)
    assert M.device_status() == 0


def test_decode_shards_padded_block_table_rows(kernel):
    # shard r's rows point into slice r of the shared cache; out-of-range page ids stay
    # out of range (flagged, not read from another shard's slice)
    w = synth.make_custom(2, 16, 1, [40, 40], 16, 2, seed=12)
    step = _gpu_shards(w)
    base = w.num_blocks
    bt = step.block_table_all.clone()
    assert int(bt[2:].max()) >= base                     # shard 1 rows are offset
    step.block_table_all[3, 0] = -5                      # shard 1, request 1, keys 0..15
    step.run()
    torch.cuda.synchronize()
    assert M.device_status() & 1
    step.block_table_all.copy_(bt)


def test_decode_without_workspace_matches(kernel):
    _check_workload(synth.make_workload("plain", lengths=[1500, 3000]), with_workspace=False)


@pytest.mark.parametrize("q_len,lengths,cp", [
    (1, [1, 2, 3], 1), (2, [1, 2], 1), (3, [1, 2, 3, 4], 2), (4, [1, 3, 5, 9], 4),
    (4, [2, 17, 33], 16), (2, [15, 16, 17], 1), (3, [63, 64, 65, 127, 128, 129], 1),
    (1, [191, 192, 193], 3), (8, [40, 300], 2), (16, [40, 300], 2), (16, [1, 17], 1),
])
@pytest.mark.parametrize("H_,bs", [(16, 16), (64, 64), (128, 64)])
def test_decode_edge_cases(q_len, lengths, cp, H_, bs, kernel):
    # a few keys per shard (down to one): outputs come close to a single |V|, where the
    # bf16 roundings of P, of a split partial and of the output approach 2e-2, so these
    # cases use the derived per-element bound of gpu_helpers (never below 2e-2)
    w = synth.make_custom(len(lengths), H_, q_len, lengths, bs, cp, base_e=(cp != 4),
                          seed=q_len * 100 + cp + H_)
    _check_workload(w, relative=True)


def _offset_16(t):
    """A copy of t whose data starts 16 bytes past a 32-byte boundary."""
    big = torch.empty(t.numel() + 32, dtype=t.dtype, device=t.device)
    base = (32 - big.data_ptr() % 32) % 32 // t.element_size()
    view = big[base + 16 // t.element_size():][:t.numel()].view(t.shape)
    view.copy_(t)
    assert view.data_ptr() % 32 == 16
    return view


@pytest.mark.parametrize("with_workspace", [True, False])
def test_decode_q_and_out_only_16_byte_aligned(with_workspace, kernel):
    # q and out need only 16-byte alignment; wider accesses must not be assumed
    w = synth.make_workload("plain", lengths=[1000, 2049])
    step = _gpu_shards(w, with_workspace)
    q16 = _offset_16(step.q)
    out16 = _offset_16(torch.zeros(step.partials[0].shape, dtype=torch.bfloat16, device=DEV))
    lse = torch.empty(step.lses[0].shape, dtype=torch.float32, device=DEV)
    M.mla_decode(q16, step.pools[0], step.block_table, step.seq_lens[0], step.gseq, step.q_len,
                 step.cp, 0, step.scale, out=out16, lse=lse, lse_base_e=step.lse_base_e,
                 workspace=step.workspace)
    torch.cuda.synchronize()
    ro, rl, _, _ = H.oracle_shards(w)
    H.compare(out16, lse, ro[0], rl[0], False, "16-byte aligned q / out")
    assert M.device_status() == 0


@pytest.mark.parametrize("B_,H_,q_len,lengths,cp,with_ws", [
    (1, 128, 4, [100], 1, True),        # 2 tiles, 4 row tiles: fewer tiles than groups
    (3, 96, 4, [700, 64, 1500], 2, True),   # 3 row tiles per request: 25 groups of 3
    (2, 48, 8, [900, 2100], 1, True),   # 3 row tiles, the last one partial
    (4, 128, 8, [40, 333, 64, 1025], 4, True),  # 8 row tiles
    (3, 96, 4, [700, 64, 1500], 2, False),  # whole requests per group, no workspace
    (2, 128, 8, [300, 2000], 1, False),
])
def test_decode_grouped_schedule(B_, H_, q_len, lengths, cp, with_ws, kernel):
    # clusters run in groups of ceil(q_len*H/128) (one cluster per row tile)
    w = synth.make_custom(B_, H_, q_len, lengths, 64, cp, base_e=True, seed=B_ * 31 + H_ + q_len)
    _check_workload(w, with_workspace=with_ws)


@pytest.mark.parametrize("with_ws,batched", [(True, True), (True, False), (False, True)])
def test_decode_many_short_segments(with_ws, batched, kernel):
    # 48 requests x 8 shards: many shard-requests with no key (1 or 2 positions over 8
    # ranks), many of one partial tile, some long; each request's tiles are preceded on the
    # split line by its start-up share, so group starts fall inside shares, inside tiles
    # and on tile boundaries, and a group may hold nothing but shares
    mix = [1, 2, 7, 63, 64, 65, 129, 640, 2000, 513, 8, 3000]
    lengths = [mix[(7 * i) % len(mix)] for i in range(48)]
    w = synth.make_custom(48, 128, 4, lengths, 64, 8, base_e=True, seed=4801)
    _check_workload(w, relative=True, with_workspace=with_ws, batched=batched)


def test_decode_block_table_with_wide_stride(kernel):
    w = synth.make_custom(2, 64, 2, [300, 129], 64, 2, seed=5, spare_columns=9)
    _check_workload(w)


def test_decode_bad_page_is_flagged_not_read(kernel):
    w = synth.make_custom(2, 16, 1, [40, 40], 16, 1, seed=9)
    step = _gpu_shards(w)
    bt = step.block_table.clone()
    bt[1, 1] = w.num_blocks + 1000                      # request 1, keys 16..31
    step.block_table = bt
    out, lse = step.run()
    torch.cuda.synchronize()
    assert M.device_status() & 1
    _, _, mo, ml = H.oracle_shards(w)
    H.compare(out[:1], lse[:1], mo[:1], ml[:1], what="untouched request")
    assert torch.isfinite(out[1].float()).all()


def test_decode_seq_len_beyond_table_is_flagged(kernel):
    w = synth.make_custom(1, 16, 1, [40], 16, 1, seed=10)
    step = _gpu_shards(w)
    step.seq_lens[0] = torch.tensor([10_000], dtype=torch.int32, device=DEV)
    step.gseq = torch.tensor([10_000], dtype=torch.int32, device=DEV)
    step.run()
    torch.cuda.synchronize()
    assert M.device_status() & 2                        # clamped, flagged, no fault


# ---------------------------------------------------------------------------
# full-size workloads, in the launch configuration bench.py times, sampled rows
# ---------------------------------------------------------------------------
def _sampled_full(name, sample, relative=False):
    w = synth.make_workload(name, device=DEV)
    step = step_from_workload(w, DEV)
    out, lse = step.run()
    torch.cuda.synchronize()
    assert M.device_status() == 0
    get = H.device_row_getter(w)
    outs, lses, absw, dels = [], [], [], []
    idx = [b * w.q_len + i for b, i in sample]
    for r in range(w.cp):
        o, l, a, d = H.oracle_sampled_shard(w, sample, r, get, with_abs=True)
        outs.append(o)
        lses.append(l)
        absw.append(a)
        dels.append(d)
        if r < 2 and w.cp > 1:
            H.compare(step.partials[r][idx], step.lses[r][idx], o[idx], l[idx], relative,
                      f"{name} shard {r}", a[idx], d[idx])
    mo, ml = R.ref_lse_merge(np.stack(outs), np.stack(lses), w.base_e)
    ma, _ = R.ref_lse_merge(np.stack(absw), np.stack(lses), w.base_e)
    md = np.max(np.stack(dels), axis=0)
    H.compare(out[idx], lse[idx], mo[idx], ml[idx], relative, f"{name} merged", ma[idx],
              md[idx])
    # properties that hold for every row: finite outputs, |out| bounded by max |V|
    assert torch.isfinite(out.float()).all()
    assert torch.isfinite(lse).all()


def test_full_size_plain_sampled():
    _sampled_full("plain", [(0, 0), (17, 0), (63, 0)])


def test_full_size_spec_sampled():
    _sampled_full("spec", [(0, 0), (0, 3), (31, 1)])


def test_full_size_long_sampled():
    _sampled_full("long", [(2, 0), (2, 1)], relative=True)
