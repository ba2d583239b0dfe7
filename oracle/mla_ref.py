"""Float64 CPU oracle for paged MLA decode with decode-context-parallel (DCP) shards.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this module.  It shares no code with the CUDA library and
imports nothing from the product package; the only module both sides use is ``synth``
(seeded random inputs, none of the method's arithmetic).

Everything here is the plain definition written out in float64 NumPy: pages are gathered
row by row, softmax attention is taken per (request, query row) with all heads as one
matrix, and nothing is blocked, fused or reordered beyond what the definition states.

Sources (web pages summarising three vLLM pull requests):
  [#52188] "支持 Kimi-K3 DSpark 推测解码与 DCP 并行组合" (prhub.com.cn, vLLM PR 52188)
  [#54012] "带 DCP 的 MLA decode 改用 FlashInfer 原生 CP mask" (vLLM PR 54012)
  [#48180] "为 TokenSpeed MLA 后端添加 DCP 与 Eagle 支持" (vLLM PR 48180)

Readings of points the pages leave open:
  * PAD_SLOT_ID is -1; a negative position means "rejected" and maps to PAD.
  * Query/KV head dim 576 = 512 latent + 64 rope; V is the first 512 dims of each row.
  * A query row with no visible key gets out = 0 and lse = -inf; a merge gives such a
    shard weight 0, and a merge of only empty shards gives out = 0, lse = -inf.
  * ``seq_lens[b]`` is the shard-local count for the full global length G_b; a row reads
    min(seq_lens[b], local visible length), so it never reads past seq_lens.
"""
from __future__ import annotations

import math
from typing import Callable, Optional, Sequence

import numpy as np

PAD_SLOT_ID = -1
D_V = 512
LN2 = math.log(2.0)


# ---------------------------------------------------------------------------
# Visible lengths
# ---------------------------------------------------------------------------
def ref_row_global_prefix(G, q_len: int, causal: bool = True) -> np.ndarray:
    """Global visible prefix of each row of a q_len query block.

    [#52188] section "关键源码片段", flashinfer_mla.py ``_prepare_flattened_decode_metadata``:
    in the causal branch row r of the block sees dcp_tot_seq_lens - (query_len - 1 - r),
    clamped at 0; in the non-causal branch (a DSpark draft block) every row sees the
    same context, the request's whole length.  Returns int64 [..., q_len].
    """
    G = np.asarray(G, dtype=np.int64)
    if not causal:
        return np.repeat(G[..., None], q_len, axis=-1)
    offs = np.arange(q_len - 1, -1, -1, dtype=np.int64)
    return np.maximum(G[..., None] - offs, 0)


def ref_owned_positions(G_row: int, cp: int, rank: int, interleave: int = 1) -> np.ndarray:
    """Global positions g < G_row that shard ``rank`` holds, in increasing order: the
    sequence is cut into segments of ``interleave`` positions dealt round-robin to the
    cp ranks, so g belongs to rank (g // interleave) mod cp ([#52188] section
    "关键源码片段", cp_local_slot: the segment number modulo CP_SIZE decides the owner).
    The k-th of them is the shard's local position k."""
    g = np.arange(int(G_row), dtype=np.int64)
    return g[(g // interleave) % cp == rank]


def ref_local_len(G_row, cp: int, rank: int, interleave: int = 1) -> np.ndarray:
    """Shard-local share of a global visible length under round-robin KV sharding.

    [#52188] same snippet: span = cp * interleave; local = G // span * interleave +
    clamp(G mod span - rank * interleave, 0, interleave).
    """
    G_row = np.asarray(G_row, dtype=np.int64)
    span = cp * interleave
    rem = np.clip(G_row % span - rank * interleave, 0, interleave)
    return G_row // span * interleave + rem


# ---------------------------------------------------------------------------
# Slot mapping
# ---------------------------------------------------------------------------
def ref_cp_local_slot(positions, block_table, block_size: int, cp_size: int, cp_rank: int,
                      interleave: int = 1) -> np.ndarray:
    """Shard-local KV slot of each position, PAD_SLOT_ID where this rank does not own it.

    [#52188] section "关键源码片段", cp_utils.py ``cp_local_slot``: a virtual block spans
    block_size * CP_SIZE global positions; the offset in it is split into interleave-long
    segments dealt round-robin to the ranks; an owned offset becomes
    (offset // (interleave*CP_SIZE)) * interleave + offset % interleave inside the page
    ``block_numbers``.  [#52188] section "实现拆解" step 4: the page is
    block_table[ctx_pos // (block_size * CP_SIZE)].  A negative position (rejected draft
    suffix, [#52188] section "实现拆解" step 5) gives PAD.  A non-negative position whose
    virtual block lies past the table raises ValueError.
    """
    pos = np.asarray(positions, dtype=np.int64)
    bt = np.asarray(block_table, dtype=np.int64)
    assert pos.ndim == 2 and bt.ndim == 2 and bt.shape[0] == pos.shape[0]
    out = np.full(pos.shape, PAD_SLOT_ID, dtype=np.int64)
    vbs = block_size * cp_size
    for b in range(pos.shape[0]):
        for n in range(pos.shape[1]):
            p = int(pos[b, n])
            if p < 0:
                continue
            vb = p // vbs
            if vb >= bt.shape[1]:
                raise ValueError(f"position {p} lies in virtual block {vb} >= {bt.shape[1]}")
            bn = int(bt[b, vb])
            off = p % vbs
            if cp_size == 1:
                out[b, n] = bn * block_size + off
                continue
            if (off // interleave) % cp_size != cp_rank:
                continue
            local = (off // (interleave * cp_size)) * interleave + off % interleave
            out[b, n] = bn * block_size + local
    return out


def ref_scatter_kv(pool, positions, kv_new, block_table, block_size: int, cp_size: int,
                   cp_rank: int, interleave: int = 1) -> np.ndarray:
    """Writes new KV rows into shard ``cp_rank``'s paged pool: row kv_new[b, n] goes to
    slot ref_cp_local_slot(positions)[b, n] when this rank owns that position, and
    nowhere otherwise ([#52188] section "实现拆解" step 4: the draft inputs apply
    cp_local_slot to their context and query slots, with the page of a position taken
    from block_table[pos // (block_size * CP_SIZE)], so that a rank never writes slots
    another rank is responsible for).  pool [num_blocks, block_size, D] is copied, not
    changed; the copy is returned."""
    out = np.array(pool, dtype=np.float64, copy=True)
    flat = out.reshape(-1, out.shape[-1])
    slots = ref_cp_local_slot(positions, block_table, block_size, cp_size, cp_rank, interleave)
    new = np.asarray(kv_new, dtype=np.float64)
    for b in range(slots.shape[0]):
        for n in range(slots.shape[1]):
            sl = int(slots[b, n])
            if sl != PAD_SLOT_ID:
                flat[sl] = new[b, n]
    return out


def ref_build_pool(kv_rows: Sequence[np.ndarray], block_table, block_size: int, cp: int,
                   rank: int, num_blocks: int, interleave: int = 1) -> np.ndarray:
    """Shard ``rank``'s paged pool [num_blocks, block_size, D]: every global row g of
    request b is written at ref_cp_local_slot(g) when this rank owns it; all other slots
    are NaN."""
    D = kv_rows[0].shape[1]
    pool = np.full((num_blocks * block_size, D), np.nan, dtype=np.float64)
    for b, rows in enumerate(kv_rows):
        G = rows.shape[0]
        pos = np.arange(G, dtype=np.int64).reshape(1, G)
        slots = ref_cp_local_slot(pos, np.asarray(block_table)[b:b + 1], block_size, cp, rank,
                                  interleave)[0]
        own = slots >= 0
        pool[slots[own]] = np.asarray(rows, dtype=np.float64)[own]
    return pool.reshape(num_blocks, block_size, D)


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------
def _softmax_attend(q_rows: np.ndarray, keys: np.ndarray, scale: float):
    """softmax(scale * q K^T) V over all keys, V = keys[:, :512].  Returns (out, lse_e)."""
    s = scale * (q_rows @ keys.T)                  # [H, L]
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    denom = e.sum(axis=1, keepdims=True)
    lse = m[:, 0] + np.log(denom[:, 0])
    p = e / denom
    return p @ keys[:, :D_V], lse


def ref_abs_weighted(q, kv_rows, G, q_len: int, cp_world: int, cp_rank: int, scale: float,
                     rows=None, row_getter=None, interleave: int = 1, causal: bool = True):
    """Error scale of a softmax-weighted sum, not a result: sum_l softmax(s)_l |V_l| per
    (row, head, dim) over the keys shard ``cp_rank`` holds (same visibility as
    ref_mla_decode_global).  A kernel that rounds the softmax weights to bf16 (8
    significant bits, round to nearest) perturbs each weight by at most 2^-9 of itself,
    so its output error is bounded by 2^-9 times this quantity; shards combine it with
    the same LSE weights as their outputs."""
    q = np.asarray(q)
    B, ql, H, D = q.shape
    G = np.asarray(G, dtype=np.int64)
    out = np.zeros((B * q_len, H, D_V), dtype=np.float64)
    todo = rows if rows is not None else [(b, i) for b in range(B) for i in range(q_len)]
    for b, i in todo:
        Gi = int(ref_row_global_prefix(G[b], q_len, causal)[i])
        idx = ref_owned_positions(Gi, cp_world, cp_rank, interleave)
        if idx.size == 0:
            continue
        keys = (row_getter(b, idx) if row_getter is not None
                else np.asarray(kv_rows[b], dtype=np.float64)[idx])
        keys = np.asarray(keys, dtype=np.float64)
        s = scale * (np.asarray(q[b, i], dtype=np.float64) @ keys.T)
        e = np.exp(s - s.max(axis=1, keepdims=True))
        out[b * q_len + i] = (e / e.sum(axis=1, keepdims=True)) @ np.abs(keys[:, :D_V])
    return out


def ref_gather_pages(kv_cache, block_table_row, L: int) -> np.ndarray:
    """Rows 0..L-1 of one request's shard-local sequence: local position l lives at
    page block_table_row[l // block_size], offset l % block_size ([#54012] section
    "关键源码片段": block_tables/seq_lens handed to the kernel)."""
    bs = kv_cache.shape[1]
    npages = (L + bs - 1) // bs
    ids = np.asarray(block_table_row[:npages], dtype=np.int64)
    rows = np.asarray(kv_cache[ids], dtype=np.float64).reshape(npages * bs, -1)
    return rows[:L]


def ref_mla_decode(q, kv_cache, block_table, seq_lens, causal_seqlens_global, q_len: int,
                   cp_world: int, cp_rank: int, scale: float, lse_base_e: bool = True,
                   rows: Optional[Sequence[tuple]] = None, interleave: int = 1,
                   causal: bool = True):
    """One shard's partial MLA decode over its paged latent cache.

    q [B, q_len, H, 576]; kv_cache [num_blocks, block_size, 576]; block_table [B, *];
    seq_lens [B] shard-local counts; causal_seqlens_global [B] (None only when
    cp_world == 1 or the block is non-causal).
    Causal: row i of request b sees global prefix G_i ([#52188] snippet), of which this
    shard holds L_i = min(seq_lens[b], local_len(G_i)) under round-robin segments of
    ``interleave`` positions ([#52188] snippet: span = cp * interleave, remainder
    clamp; [#54012] section "实现拆解" step 3: the kernel masks by global position with
    cp_world/cp_rank).  Non-causal (a DSpark draft block, [#52188] snippet's other
    branch: seq_lens repeated per query row): every row sees the shard's whole local
    sequence, L_i = seq_lens[b].  Returns out [B*q_len, H, 512] and lse [B*q_len, H]
    in base e, or base 2 when lse_base_e is False ([#48180] section "实现拆解" step 1:
    LSE returned in log2).  ``rows`` limits the work to the listed (b, i) pairs; the
    other outputs stay 0 / -inf.
    """
    q = np.asarray(q)
    B, ql, H, D = q.shape
    assert ql == q_len
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    if causal_seqlens_global is None:
        if cp_world != 1 and causal:
            raise ValueError("causal_seqlens_global is required when cp_world > 1")
        G = seq_lens
    else:
        G = np.asarray(causal_seqlens_global, dtype=np.int64)
    out = np.zeros((B * q_len, H, D_V), dtype=np.float64)
    lse = np.full((B * q_len, H), -np.inf, dtype=np.float64)
    todo = rows if rows is not None else [(b, i) for b in range(B) for i in range(q_len)]
    for b, i in todo:
        if causal:
            Gi = int(ref_row_global_prefix(G[b], q_len)[i])
            Li = min(int(seq_lens[b]), int(ref_local_len(Gi, cp_world, cp_rank, interleave)))
        else:
            Li = int(seq_lens[b])
        if Li == 0:
            continue
        keys = ref_gather_pages(kv_cache, np.asarray(block_table)[b], Li)
        o, l_e = _softmax_attend(np.asarray(q[b, i], dtype=np.float64), keys, scale)
        out[b * q_len + i] = o
        lse[b * q_len + i] = l_e if lse_base_e else l_e / LN2
    return out, lse


def ref_mla_decode_global(q, kv_rows: Sequence[np.ndarray], G, q_len: int, cp_world: int,
                          cp_rank: int, scale: float, lse_base_e: bool = True,
                          rows: Optional[Sequence[tuple]] = None,
                          row_getter: Optional[Callable] = None, interleave: int = 1,
                          causal: bool = True):
    """The same shard result stated on global positions, with no pages: shard ``cp_rank``
    holds global position g iff (g // interleave) mod cp_world == cp_rank, and row i
    sees g < G_i (causal) or g < G_b (non-causal).  ``row_getter(b, idx)`` may supply
    rows lazily (large cases).
    """
    q = np.asarray(q)
    B, ql, H, D = q.shape
    G = np.asarray(G, dtype=np.int64)
    out = np.zeros((B * q_len, H, D_V), dtype=np.float64)
    lse = np.full((B * q_len, H), -np.inf, dtype=np.float64)
    todo = rows if rows is not None else [(b, i) for b in range(B) for i in range(q_len)]
    for b, i in todo:
        Gi = int(ref_row_global_prefix(G[b], q_len, causal)[i])
        idx = ref_owned_positions(Gi, cp_world, cp_rank, interleave)
        if idx.size == 0:
            continue
        keys = (row_getter(b, idx) if row_getter is not None
                else np.asarray(kv_rows[b], dtype=np.float64)[idx])
        o, l_e = _softmax_attend(np.asarray(q[b, i], dtype=np.float64),
                                 np.asarray(keys, dtype=np.float64), scale)
        out[b * q_len + i] = o
        lse[b * q_len + i] = l_e if lse_base_e else l_e / LN2
    return out, lse


def ref_attention_global(q, kv_rows: Sequence[np.ndarray], G, q_len: int, scale: float,
                         rows: Optional[Sequence[tuple]] = None,
                         row_getter: Optional[Callable] = None, causal: bool = True):
    """Unsharded, unpaged ground truth: row i of request b attends to global rows
    g < G_b - (q_len - 1 - i), or g < G_b when the block is non-causal.
    Returns (out, lse_e)."""
    return ref_mla_decode_global(q, kv_rows, G, q_len, 1, 0, scale, True, rows, row_getter,
                                 1, causal)


# ---------------------------------------------------------------------------
# LSE merge
# ---------------------------------------------------------------------------
def ref_lse_merge(partials, lses, lse_base_e: bool = True):
    """Merge n shards' (out, lse) into the full result.

    [#54012] section "实现拆解" step 3 and [#48180] section "实现拆解" step 2: every shard
    returns a partial output and an LSE in one common base, and the shards are combined
    through those LSEs.  With M = max_s lse_s and w_s = base**(lse_s - M):
    out = sum_s w_s o_s / sum_s w_s, lse = M + log_base(sum_s w_s).
    partials [n, T, H, Dv], lses [n, T, H]; all-empty rows give out 0, lse -inf.
    """
    P = np.asarray(partials, dtype=np.float64)
    L = np.asarray(lses, dtype=np.float64)
    M = L.max(axis=0)                                  # [T, H]
    empty = np.isneginf(M)
    Ms = np.where(empty, 0.0, M)
    if lse_base_e:
        w = np.exp(L - Ms[None])
    else:
        w = np.exp2(L - Ms[None])
    w = np.where(np.isneginf(L), 0.0, w)
    wsum = w.sum(axis=0)
    safe = np.where(empty, 1.0, wsum)
    out = (w[..., None] * P).sum(axis=0) / safe[..., None]
    out[empty] = 0.0
    lse = Ms + (np.log(safe) if lse_base_e else np.log2(safe))
    lse[empty] = -np.inf
    return out, lse
