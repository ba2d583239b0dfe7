"""Plant plausible mistakes in the oracle (CPU only) and check that the pins notice.

Each mutation replaces one oracle function with a subtly wrong version; the test passes
only if at least one of the pin checks then fails.  This shows that the pins are not
restatements of the oracle's own formulas.
"""
import math

import numpy as np
import pytest

import oracle.mla_ref as R
import oracle_pins as P


_orig_prefix = R.ref_row_global_prefix


def _prefix_reversed(G, q_len, causal=True):
    if not causal:
        return _orig_prefix(G, q_len, False)
    G = np.asarray(G, dtype=np.int64)
    return np.maximum(G[..., None] - np.arange(q_len, dtype=np.int64), 0)


def _prefix_unclamped(G, q_len, causal=True):
    if not causal:
        return _orig_prefix(G, q_len, False)
    G = np.asarray(G, dtype=np.int64)
    return G[..., None] - np.arange(q_len - 1, -1, -1, dtype=np.int64)


def _prefix_off_by_one(G, q_len, causal=True):
    if not causal:
        return _orig_prefix(G, q_len, False)
    G = np.asarray(G, dtype=np.int64)
    return np.maximum(G[..., None] - np.arange(q_len, 0, -1, dtype=np.int64), 0)


def _prefix_noncausal_is_causal(G, q_len, causal=True):
    return _orig_prefix(G, q_len, True)


def _prefix_noncausal_drops_last(G, q_len, causal=True):
    if causal:
        return _orig_prefix(G, q_len, True)
    return np.maximum(_orig_prefix(G, q_len, False) - 1, 0)


_orig_owned = R.ref_owned_positions


def _owned_ignores_interleave(G_row, cp, rank, interleave=1):
    return _orig_owned(G_row, cp, rank, 1)


def _owned_rank_shift(G_row, cp, rank, interleave=1):
    return _orig_owned(G_row, cp, (rank + 1) % cp, interleave)


def _local_rank_shift(G_row, cp, rank, interleave=1):
    G_row = np.asarray(G_row, dtype=np.int64)
    span = cp * interleave
    rem = np.clip(G_row % span - (rank + 1) * interleave, 0, interleave)
    return G_row // span * interleave + rem


def _local_no_upper_clip(G_row, cp, rank, interleave=1):
    G_row = np.asarray(G_row, dtype=np.int64)
    span = cp * interleave
    rem = np.maximum(G_row % span - rank * interleave, 0)
    return G_row // span * interleave + rem


_orig_slot = R.ref_cp_local_slot


def _slot_wrong_virtual_block(positions, block_table, block_size, cp_size, cp_rank,
                              interleave=1):
    # looks up the page by pos // block_size instead of the virtual block
    pos = np.asarray(positions, dtype=np.int64)
    bt = np.asarray(block_table, dtype=np.int64)
    big = np.repeat(bt, cp_size, axis=1)
    return _orig_slot(pos, big, block_size, cp_size, cp_rank, interleave)


def _slot_ignores_interleave(positions, block_table, block_size, cp_size, cp_rank,
                             interleave=1):
    return _orig_slot(positions, block_table, block_size, cp_size, cp_rank, 1)


def _attend_v_from_tail(q_rows, keys, scale):
    s = scale * (q_rows @ keys.T)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    den = e.sum(axis=1, keepdims=True)
    return (e / den) @ keys[:, -512:], m[:, 0] + np.log(den[:, 0])


def _attend_no_scale(q_rows, keys, scale):
    s = q_rows @ keys.T
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    den = e.sum(axis=1, keepdims=True)
    return (e / den) @ keys[:, :512], m[:, 0] + np.log(den[:, 0])


def _attend_lse_drops_max(q_rows, keys, scale):
    s = scale * (q_rows @ keys.T)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    den = e.sum(axis=1, keepdims=True)
    return (e / den) @ keys[:, :512], np.log(den[:, 0])


_orig_merge = R.ref_lse_merge


def _merge_base_ignored(partials, lses, lse_base_e=True):
    return _orig_merge(partials, lses, True)


def _merge_lse_drops_max(partials, lses, lse_base_e=True):
    o, l = _orig_merge(partials, lses, lse_base_e)
    M = np.asarray(lses, dtype=np.float64).max(axis=0)
    return o, np.where(np.isneginf(l), l, l - np.where(np.isneginf(M), 0, M))


_orig_decode = R.ref_mla_decode


def _decode_noncausal_masks_causally(q, kv_cache, block_table, seq_lens, causal_seqlens_global,
                                     q_len, cp_world, cp_rank, scale, lse_base_e=True, rows=None,
                                     interleave=1, causal=True):
    G = causal_seqlens_global if causal_seqlens_global is not None else seq_lens
    if not causal and cp_world > 1 and causal_seqlens_global is None:
        G = np.asarray(seq_lens) * cp_world
    return _orig_decode(q, kv_cache, block_table, seq_lens, G, q_len, cp_world, cp_rank,
                        scale, lse_base_e, rows, interleave, True)


def _decode_interleave_ignored(q, kv_cache, block_table, seq_lens, causal_seqlens_global,
                               q_len, cp_world, cp_rank, scale, lse_base_e=True, rows=None,
                               interleave=1, causal=True):
    return _orig_decode(q, kv_cache, block_table, seq_lens, causal_seqlens_global, q_len,
                        cp_world, cp_rank, scale, lse_base_e, rows, 1, causal)


_orig_scatter = R.ref_scatter_kv


def _scatter_writes_every_rank(pool, positions, kv_new, block_table, block_size, cp_size,
                               cp_rank, interleave=1):
    out = np.array(pool, dtype=np.float64, copy=True)
    for r in range(cp_size):
        out = np.where(np.isnan(out), _orig_scatter(out, positions, kv_new, block_table,
                                                    block_size, cp_size, r, interleave), out)
    return out


def _scatter_row_shift(pool, positions, kv_new, block_table, block_size, cp_size, cp_rank,
                       interleave=1):
    return _orig_scatter(pool, positions, np.roll(np.asarray(kv_new), 1, axis=1), block_table,
                         block_size, cp_size, cp_rank, interleave)


def _gather_wrong_page(kv_cache, block_table_row, L):
    bs = kv_cache.shape[1]
    npages = (L + bs - 1) // bs
    ids = np.roll(np.asarray(block_table_row[:npages], dtype=np.int64), 1)
    return np.asarray(kv_cache[ids], dtype=np.float64).reshape(npages * bs, -1)[:L]


MUTATIONS = {
    "prefix_reversed": ("ref_row_global_prefix", _prefix_reversed),
    "prefix_unclamped": ("ref_row_global_prefix", _prefix_unclamped),
    "prefix_off_by_one": ("ref_row_global_prefix", _prefix_off_by_one),
    "local_rank_shift": ("ref_local_len", _local_rank_shift),
    "local_no_upper_clip": ("ref_local_len", _local_no_upper_clip),
    "slot_wrong_virtual_block": ("ref_cp_local_slot", _slot_wrong_virtual_block),
    "slot_ignores_interleave": ("ref_cp_local_slot", _slot_ignores_interleave),
    "v_from_tail": ("_softmax_attend", _attend_v_from_tail),
    "no_scale": ("_softmax_attend", _attend_no_scale),
    "lse_drops_max": ("_softmax_attend", _attend_lse_drops_max),
    "merge_base_ignored": ("ref_lse_merge", _merge_base_ignored),
    "merge_lse_drops_max": ("ref_lse_merge", _merge_lse_drops_max),
    "gather_wrong_page": ("ref_gather_pages", _gather_wrong_page),
    "noncausal_is_causal": ("ref_row_global_prefix", _prefix_noncausal_is_causal),
    "noncausal_drops_last": ("ref_row_global_prefix", _prefix_noncausal_drops_last),
    "owned_ignores_interleave": ("ref_owned_positions", _owned_ignores_interleave),
    "owned_rank_shift": ("ref_owned_positions", _owned_rank_shift),
    "decode_noncausal_masks_causally": ("ref_mla_decode", _decode_noncausal_masks_causally),
    "decode_interleave_ignored": ("ref_mla_decode", _decode_interleave_ignored),
    "scatter_writes_every_rank": ("ref_scatter_kv", _scatter_writes_every_rank),
    "scatter_row_shift": ("ref_scatter_kv", _scatter_row_shift),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(R, attr, fn)
    failed = []
    for check in P.ALL_CHECKS:
        try:
            check()
        except (AssertionError, ValueError, IndexError):
            failed.append(check.__name__)
    assert failed, f"no pin noticed mutation {name}"
