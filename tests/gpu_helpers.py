"""Shared helpers of the GPU parity tests: the oracle side of a synth workload, and the
element-wise comparisons with the tolerances of the decode contract.

Tolerances: bf16 outputs within max-abs 2e-2 of the float64 oracle; fp32 LSEs within
1e-3 absolute.  The long-context workload (1% of KV rows x20) has outputs of size tens,
where one bf16 rounding alone is up to 2^-8 of the value, so an absolute 2e-2 cannot
hold for any bf16 result.  Its output bound is derived from the arithmetic, per element
(row, head, dim), with A = sum_l softmax(s)_l |V_l| (the oracle's ref_abs_weighted):

  * bf16 rounding, relative error <= u16 = 2^-8 (8 significant bits, round to nearest
    even), happens four times on the way to a merged output: the softmax weights P fed to
    the PV MMA (error <= u16 * A), a unit's split partial, the shard partial, the merged
    output (each <= u16 * A, since |partial| <= its own A and the merge weights the A's
    the same way);
  * scores: 576 exact bf16 products summed by tcgen05.mma in 36 instructions of 16
    products each into an fp32 accumulator.  Whatever order an instruction sums its 16
    products in, the first-order error bound of a sum of n terms is (n-1) u |terms|, so
    one instruction adds at most 15 u sum|products of its block| and the 36 accumulations
    at most 35 u sum|products|: delta <= 50 u scale sum_d |q_d k_d| per key, doubled to
    cover truncation instead of rounding (u = 2^-24), 100 u in all.  A weight moves by
    at most e^{+-delta} relative to the others, the output by at most 2 (e^delta - 1) A.

  |gpu - ref| <= 2e-2 + (4 * 2^-8 + 2 (e^delta - 1)) * A,
  delta = 100 * 2^-24 * scale * max_l sum_d |q_d k_{l,d}| over the row's visible keys.

Every other workload uses max-abs 2e-2; every LSE 1e-3 absolute.  ``compare`` returns the
measured errors (absolute, and relative to the bound) and ``report`` prints them.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle.mla_ref as R

OUT_TOL = 2e-2
LSE_TOL = 1e-3


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


U_FP32 = 2.0 ** -24
U_BF16 = 2.0 ** -8
SCORE_ROUNDINGS = 100        # 2 x (15 inside one 16-product MMA + 35 accumulations)
BF16_ROUNDINGS = 4           # P, split partial, shard partial, merged output


def score_error_scale(q, key_rows, G, q_len, cp, rank, scale, rows=None, row_getter=None,
                      interleave=1, causal=True):
    """delta of the score bound per (row, head): 100·u·scale·max_l Σ_d |q_d k_{l,d}| over
    the keys shard ``rank`` holds (the visibility of ref_abs_weighted)."""
    q = np.asarray(q)
    B, ql, H, D = q.shape
    out = np.zeros((B * q_len, H), dtype=np.float64)
    todo = rows if rows is not None else [(b, i) for b in range(B) for i in range(q_len)]
    for b, i in todo:
        Gi = int(R.ref_row_global_prefix(int(G[b]), q_len, causal)[i])
        idx = R.ref_owned_positions(Gi, cp, rank, interleave)
        if idx.size == 0:
            continue
        keys = (row_getter(b, idx) if row_getter is not None
                else np.asarray(key_rows[b], dtype=np.float64)[idx])
        t = np.abs(np.asarray(q[b, i], dtype=np.float64)) @ np.abs(np.asarray(keys, np.float64)).T
        out[b * q_len + i] = SCORE_ROUNDINGS * U_FP32 * scale * t.max(axis=1)
    return out


def out_bound(out_ref, relative=False, abs_weighted=None, score_delta=None):
    """Per-element bound on |gpu - ref| of the decode contract (see the module doc)."""
    if not relative:
        return np.full(out_ref.shape, OUT_TOL)
    assert abs_weighted is not None and score_delta is not None
    k = BF16_ROUNDINGS * U_BF16 + 2.0 * np.expm1(np.asarray(score_delta))[..., None]
    return OUT_TOL + k * abs_weighted


def compare(out_gpu, lse_gpu, out_ref, lse_ref, relative=False, what="", abs_weighted=None,
            score_delta=None):
    """Asserts the decode contract's tolerances element by element; returns (worst
    absolute error, worst LSE error, worst error as a fraction of its bound)."""
    og = f64(out_gpu) if isinstance(out_gpu, torch.Tensor) else np.asarray(out_gpu, np.float64)
    lg = f64(lse_gpu) if isinstance(lse_gpu, torch.Tensor) else np.asarray(lse_gpu, np.float64)
    assert og.shape == out_ref.shape, (og.shape, out_ref.shape)
    assert np.all(np.isfinite(og)), f"{what}: non-finite output"
    err = np.abs(og - out_ref)
    bound = out_bound(out_ref, relative, abs_weighted, score_delta)
    frac = err / bound
    worst_frac = float(frac.max()) if frac.size else 0.0
    worst = float(err.max()) if err.size else 0.0
    assert worst_frac <= 1.0, (f"{what}: out error {worst:.3e} exceeds its bound "
                               f"({worst_frac:.2f} of it)")
    fin = np.isfinite(lse_ref)
    assert np.array_equal(fin, np.isfinite(lg)), f"{what}: -inf pattern of lse differs"
    assert np.all(lg[~fin] == -np.inf), f"{what}: empty rows must have lse -inf"
    lerr = float(np.abs(lg[fin] - lse_ref[fin]).max()) if fin.any() else 0.0
    assert lerr <= LSE_TOL, f"{what}: lse error {lerr:.3e} > {LSE_TOL}"
    report(what, worst, lerr, worst_frac, abs_weighted, err)
    return worst, lerr, worst_frac


def report(what, worst, lerr, worst_frac, abs_weighted=None, err=None):
    """Prints the measured errors of one comparison (pytest shows them with -s or -rA)."""
    extra = ""
    if abs_weighted is not None and err is not None and err.size:
        extra = f"  max |err|/A {float((err / np.maximum(abs_weighted, 1e-30)).max()):.3e}"
    print(f"[parity] {what}: max|out err| {worst:.3e}  max|lse err| {lerr:.3e}  "
          f"bound used {worst_frac:.3f}{extra}")


def oracle_workload_rows(w):
    q = f64(w.q)
    rows = [f64(w.rows_of(b)) for b in range(w.B)]
    return q, rows


def oracle_shards(w, with_abs=False):
    """Per-shard (out, lse) over oracle-built pools, plus the merged result; with
    ``with_abs`` also the per-shard and merged ref_abs_weighted error scales and the
    per-shard and merged score deltas of rule (3)."""
    q, rows = oracle_workload_rows(w)
    bt = w.block_table.numpy()
    G = w.G.numpy()
    outs, lses, absw, dels = [], [], [], []
    il, causal = w.interleave, w.causal
    for r in range(w.cp):
        pool = R.ref_build_pool(rows, bt, w.bs, w.cp, r, w.num_blocks, il)
        sl = R.ref_local_len(G, w.cp, r, il)
        o, l = R.ref_mla_decode(q, pool, bt, sl, G if w.cp > 1 else None, w.q_len, w.cp, r,
                                w.scale, w.base_e, interleave=il, causal=causal)
        outs.append(o)
        lses.append(l)
        if with_abs:
            absw.append(R.ref_abs_weighted(q, rows, G, w.q_len, w.cp, r, w.scale,
                                           interleave=il, causal=causal))
            dels.append(score_error_scale(q, rows, G, w.q_len, w.cp, r, w.scale,
                                          interleave=il, causal=causal))
    mo, ml = R.ref_lse_merge(np.stack(outs), np.stack(lses), w.base_e)
    if not with_abs:
        return outs, lses, mo, ml
    ma, _ = R.ref_lse_merge(np.stack(absw), np.stack(lses), w.base_e)
    md = np.max(np.stack(dels), axis=0)
    return outs, lses, mo, ml, absw, ma, dels, md


def device_row_getter(w):
    """getter(b, idx) -> float64 rows idx of request b, gathered from the workload's
    (possibly device-resident) global KV rows -- the generator's draws, not a kernel
    result."""
    def get(b, idx):
        off = int(w.kv_offsets[b])
        ii = torch.from_numpy(np.asarray(idx, dtype=np.int64) + off).to(w.kv_global.device)
        return f64(w.kv_global.index_select(0, ii))
    return get


def oracle_sampled_shard(w, sample, rank, getter, with_abs=False):
    """Shard ``rank``'s result for sampled (b, i) rows, stated on global positions."""
    q = f64(w.q)
    il, causal = w.interleave, w.causal
    o, l = R.ref_mla_decode_global(q, None, w.G.numpy(), w.q_len, w.cp, rank, w.scale,
                                   w.base_e, rows=sample, row_getter=getter, interleave=il,
                                   causal=causal)
    if not with_abs:
        return o, l
    a = R.ref_abs_weighted(q, None, w.G.numpy(), w.q_len, w.cp, rank, w.scale, rows=sample,
                           row_getter=getter, interleave=il, causal=causal)
    d = score_error_scale(q, None, w.G.numpy(), w.q_len, w.cp, rank, w.scale, rows=sample,
                          row_getter=getter, interleave=il, causal=causal)
    return o, l, a, d
