"""Shared helpers of the GPU parity tests: the oracle side of a synth workload, and the
element-wise comparisons with the tolerances of the decode contract.

Tolerances: bf16 outputs within max-abs 2e-2 of the float64 oracle; fp32 LSEs within
1e-3 absolute.  For the long-context workload (1% of KV rows x20, so |out| reaches tens)
the output bound is per element
    |gpu - ref| <= 2e-2 * max(1, |ref|) + 2^-8 * A,   A = sum_l softmax(s)_l |V_l|,
because (1) a bf16 result there has a half-ulp of up to 0.125, so an absolute 2e-2
cannot hold even for a correctly rounded value, and (2) the tensor-core PV product takes
the softmax weights in bf16, which moves each weight by up to 2^-9 of itself: with a few
x20 keys sharing the weight, an output element near zero can be a difference of terms
of size ~50, whose bf16-weight error (bounded by 2^-9 A) exceeds 2e-2 although every
step is correctly rounded.  A is computed by the oracle (ref_abs_weighted); a wrong key
or a wrong weight moves the result by O(|V|), far above 2^-8 A.  (3) The scores are
fp32 sums of 576 products.  A floating-point sum of n terms is within n·u·Σ|terms| of
the exact sum (u = 2^-24, the fp32 unit roundoff), so a weight moves by a factor
e^{±δ} with δ = 576·u·scale·max_l Σ_d |q_d k_{l,d}|, and the output by at most
2(e^δ − 1)·A.  With x20 keys Σ|q k| reaches ~10^4 and this term reaches a few 10^-2 A;
for N(0,1) keys it is ~10^-3 A.  The bound used is therefore
    |gpu - ref| <= 2e-2 * max(1, |ref|) + (2^-8 + 2(e^δ - 1)) * A.
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


def score_error_scale(q, key_rows, G, q_len, cp, rank, scale, rows=None, row_getter=None):
    """delta of rule (3) per (row, head): 576·u·scale·max_l Σ_d |q_d k_{l,d}| over the
    keys shard ``rank`` holds (the visibility of ref_abs_weighted)."""
    q = np.asarray(q)
    B, ql, H, D = q.shape
    out = np.zeros((B * q_len, H), dtype=np.float64)
    todo = rows if rows is not None else [(b, i) for b in range(B) for i in range(q_len)]
    for b, i in todo:
        Gi = max(0, int(G[b]) - (q_len - 1 - i))
        idx = np.arange(rank, Gi, cp, dtype=np.int64)
        if idx.size == 0:
            continue
        keys = (row_getter(b, idx) if row_getter is not None
                else np.asarray(key_rows[b], dtype=np.float64)[idx])
        t = np.abs(np.asarray(q[b, i], dtype=np.float64)) @ np.abs(np.asarray(keys, np.float64)).T
        out[b * q_len + i] = D * U_FP32 * scale * t.max(axis=1)
    return out


def compare(out_gpu, lse_gpu, out_ref, lse_ref, relative=False, what="", abs_weighted=None,
            score_delta=None):
    og = f64(out_gpu)
    lg = f64(lse_gpu)
    assert og.shape == out_ref.shape, (og.shape, out_ref.shape)
    assert np.all(np.isfinite(og)), f"{what}: non-finite output"
    err = np.abs(og - out_ref)
    if relative:
        assert abs_weighted is not None
        k = 2.0 ** -8
        if score_delta is not None:
            k = k + 2.0 * np.expm1(np.asarray(score_delta))[..., None]
        err = err / (np.maximum(1.0, np.abs(out_ref)) + abs_weighted * k / OUT_TOL)
    worst = float(err.max()) if err.size else 0.0
    assert worst <= OUT_TOL, f"{what}: out error {worst:.3e} > {OUT_TOL}"
    fin = np.isfinite(lse_ref)
    assert np.array_equal(fin, np.isfinite(lg)), f"{what}: -inf pattern of lse differs"
    assert np.all(lg[~fin] == -np.inf), f"{what}: empty rows must have lse -inf"
    lerr = float(np.abs(lg[fin] - lse_ref[fin]).max()) if fin.any() else 0.0
    assert lerr <= LSE_TOL, f"{what}: lse error {lerr:.3e} > {LSE_TOL}"
    return worst, lerr


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
    for r in range(w.cp):
        pool = R.ref_build_pool(rows, bt, w.bs, w.cp, r, w.num_blocks)
        sl = R.ref_local_len(G, w.cp, r)
        o, l = R.ref_mla_decode(q, pool, bt, sl, G if w.cp > 1 else None, w.q_len, w.cp, r,
                                w.scale, w.base_e)
        outs.append(o)
        lses.append(l)
        if with_abs:
            absw.append(R.ref_abs_weighted(q, rows, G, w.q_len, w.cp, r, w.scale))
            dels.append(score_error_scale(q, rows, G, w.q_len, w.cp, r, w.scale))
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
    o, l = R.ref_mla_decode_global(q, None, w.G.numpy(), w.q_len, w.cp, rank, w.scale,
                                   w.base_e, rows=sample, row_getter=getter)
    if not with_abs:
        return o, l
    a = R.ref_abs_weighted(q, None, w.G.numpy(), w.q_len, w.cp, rank, w.scale, rows=sample,
                           row_getter=getter)
    d = score_error_scale(q, None, w.G.numpy(), w.q_len, w.cp, rank, w.scale, rows=sample,
                          row_getter=getter)
    return o, l, a, d
