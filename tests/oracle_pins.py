"""Checks that pin the float64 oracle to facts other than itself.

Each ``check_*`` raises AssertionError on a mismatch.  ``test_oracle_pins.py`` runs them
on the oracle as written; ``test_oracle_mutations.py`` plants plausible mistakes in the
oracle (on the CPU) and asserts that at least one check then fails.

What pins what:
  * hand-derived fixtures (tests/golden/*.txt) pin the slot mapping and the per-row
    visible lengths to the definitions on the pages;
  * brute-force counting of owned positions pins the round-robin local length;
  * torch's float64 scaled_dot_product_attention with a position-id causal mask pins
    the decode (textbook causal attention, MQA broadcast over heads);
  * a pure-Python triple loop pins the decode on tiny inputs;
  * closed forms pin the LSE merge (split softmax == full softmax) and the bases;
  * merging per-shard results over oracle-built pools == unsharded attention pins the
    sharding, the paging and the merge together.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import oracle.mla_ref as R

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _parse_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([[int(x) for x in part.split()] for part in line.split("|")])
    return rows


def _bf16(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).to(torch.float64).numpy()


def make_small_case(seed, B, H, q_len, G, bs, D=576):
    g = torch.Generator().manual_seed(seed)
    q = _bf16(torch.randn(B, q_len, H, D, generator=g))
    rows = [_bf16(torch.randn(int(n), D, generator=g)) for n in G]
    return q, rows


def make_block_table(seed, B, pages_per_req, extra=1):
    g = torch.Generator().manual_seed(seed + 77)
    total = B * pages_per_req
    perm = torch.randperm(total, generator=g).numpy().astype(np.int64)
    bt = np.full((B, pages_per_req + extra), total, dtype=np.int64)   # spare page id
    bt[:, :pages_per_req] = perm.reshape(B, pages_per_req)
    return bt, total + 1


# ---------------------------------------------------------------------------
def check_slot_golden():
    bt = np.array([[5, 9]], dtype=np.int64)
    for (cp, il, rank), pos, want in _parse_golden("cp_local_slot_hand.txt"):
        got = R.ref_cp_local_slot(np.array([pos]), bt, 4, cp, rank, il)[0]
        assert list(got) == want, (cp, il, rank, list(got), want)


def check_local_len_golden():
    for (G, q_len, cp, rank), prefix, local in _parse_golden("local_len_hand.txt"):
        pr = R.ref_row_global_prefix(G, q_len)
        assert list(pr) == prefix, (G, q_len, list(pr), prefix)
        ll = R.ref_local_len(pr, cp, rank, 1)
        assert list(ll) == local, (G, q_len, cp, rank, list(ll), local)


def check_local_len_bruteforce():
    """Count owned global positions one by one: position g belongs to rank
    (g // interleave) mod cp (round-robin segments of ``interleave`` positions)."""
    for cp in (1, 2, 3, 8):
        for il in (1, 2, 4):
            span = cp * il
            for rank in range(cp):
                for G in range(0, 3 * span + 5):
                    want = sum(1 for g in range(G) if (g // il) % cp == rank)
                    got = int(R.ref_local_len(G, cp, rank, il))
                    assert got == want, (cp, il, rank, G, got, want)


def check_row_prefix_positions():
    """Row i of a q_len block is the token at absolute position G - q_len + i; causal
    attention lets it see every key at a position <= its own."""
    for G in range(0, 12):
        for q_len in range(1, 6):
            got = R.ref_row_global_prefix(G, q_len)
            for i in range(q_len):
                pos = G - q_len + i
                want = max(0, pos + 1)
                assert int(got[i]) == want, (G, q_len, i, int(got[i]), want)


def check_slot_bruteforce():
    """Within each virtual block the owned positions, taken in increasing order, fill
    local offsets 0, 1, 2, ... of the page; across ranks the owned (rank, slot) pairs
    cover every slot of every page exactly once; rejected positions give PAD."""
    rng = np.random.default_rng(5)
    for bs, cp, il in [(4, 2, 1), (8, 4, 2), (16, 2, 1), (6, 3, 2), (4, 1, 1), (16, 8, 1)]:
        nvb = 5
        bt = rng.permutation(50)[:nvb].reshape(1, nvb)
        pos = np.arange(nvb * bs * cp).reshape(1, -1)
        seen = {}
        for rank in range(cp):
            slots = R.ref_cp_local_slot(pos, bt, bs, cp, rank, il)[0]
            for vb in range(nvb):
                k = 0
                for p in range(vb * bs * cp, (vb + 1) * bs * cp):
                    owner = (p // il) % cp
                    s = int(slots[p])
                    if owner != rank:
                        assert s == R.PAD_SLOT_ID, (bs, cp, il, rank, p, s)
                        continue
                    assert s == int(bt[0, vb]) * bs + k, (bs, cp, il, rank, p, s, k)
                    k += 1
                    assert (rank, s) not in seen
                    seen[(rank, s)] = p
                assert k == bs, (bs, cp, il, rank, vb, k)
        assert len(seen) == cp * nvb * bs
        rej = R.ref_cp_local_slot(np.array([[-1, -7, 0]]), bt, bs, cp, 0, il)[0]
        assert rej[0] == R.PAD_SLOT_ID and rej[1] == R.PAD_SLOT_ID


def _sdpa_reference(q_np, rows, G, q_len, scale):
    """torch float64 SDPA, one request at a time, MQA broadcast (1 KV head, H query
    heads), causal mask from position ids."""
    outs, lses = [], []
    B, _, H, D = q_np.shape
    for b in range(B):
        K = torch.from_numpy(np.asarray(rows[b][:G[b]], dtype=np.float64))
        Q = torch.from_numpy(np.asarray(q_np[b], dtype=np.float64))            # [q_len, H, D]
        qpos = torch.arange(G[b] - q_len, G[b])
        kpos = torch.arange(G[b])
        mask = kpos[None, :] <= qpos[:, None]                                # [q_len, G]
        Qh = Q.permute(1, 0, 2).unsqueeze(0)                                  # [1, H, q_len, D]
        Kh = K[None, None].expand(1, H, G[b], D)
        Vh = K[None, None, :, :512].expand(1, H, G[b], 512)
        o = torch.nn.functional.scaled_dot_product_attention(
            Qh, Kh, Vh, attn_mask=mask[None, None].expand(1, H, q_len, G[b]), scale=scale)
        s = (Qh @ Kh.transpose(-1, -2)) * scale
        s = s.masked_fill(~mask[None, None], float("-inf"))
        lse = torch.logsumexp(s, dim=-1)                                      # [1, H, q_len]
        outs.append(o[0].permute(1, 0, 2).numpy())
        lses.append(lse[0].permute(1, 0).numpy())
    return np.concatenate(outs, 0), np.concatenate(lses, 0)


def check_decode_vs_sdpa():
    """cp 1, paged oracle vs textbook causal attention (library SDPA, float64)."""
    for seed, (B, H, q_len, G, bs) in enumerate([(2, 8, 1, (37, 130), 16),
                                                 (2, 4, 3, (37, 130), 16),
                                                 (3, 2, 4, (5, 64, 65), 8)]):
        q, rows = make_small_case(seed, B, H, q_len, G, bs)
        ppr = max((n + bs - 1) // bs for n in G)
        bt, nb = make_block_table(seed, B, ppr)
        pool = R.ref_build_pool(rows, bt, bs, 1, 0, nb)
        scale = 1.0 / math.sqrt(192.0)
        out, lse = R.ref_mla_decode(q, pool, bt, np.array(G), None, q_len, 1, 0, scale, True)
        ro, rl = _sdpa_reference(q, rows, list(G), q_len, scale)
        assert np.max(np.abs(out - ro)) < 1e-12, np.max(np.abs(out - ro))
        assert np.max(np.abs(lse - rl)) < 1e-12, np.max(np.abs(lse - rl))


def check_decode_bruteforce_tiny():
    """Pure-Python loops with math.exp on the tiny workload's sizes (a few heads)."""
    B, H, q_len, G, bs = 2, 16, 3, (37, 130), 16
    q, rows = make_small_case(11, B, H, q_len, G, bs)
    ppr = max((n + bs - 1) // bs for n in G)
    bt, nb = make_block_table(11, B, ppr)
    pool = R.ref_build_pool(rows, bt, bs, 1, 0, nb)
    scale = 1.0 / math.sqrt(192.0)
    out, lse = R.ref_mla_decode(q, pool, bt, np.array(G), None, q_len, 1, 0, scale, True)
    for b in range(B):
        for i in range(q_len):
            vis = G[b] - (q_len - 1 - i)
            for h in (0, 7, 15):
                qv = [float(x) for x in q[b, i, h]]
                s = []
                for g in range(vis):
                    kr = rows[b][g]
                    acc = 0.0
                    for d in range(576):
                        acc += qv[d] * float(kr[d])
                    s.append(acc * scale)
                m = max(s)
                den = sum(math.exp(x - m) for x in s)
                want_lse = m + math.log(den)
                assert abs(lse[b * q_len + i, h] - want_lse) < 1e-9
                for d in (0, 1, 255, 511):
                    num = sum(math.exp(s[g] - m) * float(rows[b][g][d]) for g in range(vis))
                    assert abs(out[b * q_len + i, h, d] - num / den) < 1e-9


def check_merge_closed_form():
    """Softmax over a set split into groups: merging the groups' (out, lse) equals the
    softmax over the whole set, in base e and base 2; an empty group has lse -inf and
    weight 0; merging only empty groups gives 0 / -inf."""
    rng = np.random.default_rng(3)
    n_items, n_groups, Dv = 40, 5, 7
    s = rng.normal(size=(3, n_items)) * 4.0
    v = rng.normal(size=(n_items, Dv))
    full_m = s.max(1, keepdims=True)
    full_p = np.exp(s - full_m)
    full_out = (full_p / full_p.sum(1, keepdims=True)) @ v
    full_lse = full_m[:, 0] + np.log(full_p.sum(1))
    groups = np.array_split(rng.permutation(n_items), n_groups - 1) + [np.array([], dtype=int)]
    parts, lses = [], []
    for g in groups:
        if g.size == 0:
            parts.append(np.zeros((3, Dv)))
            lses.append(np.full(3, -np.inf))
            continue
        gm = s[:, g].max(1, keepdims=True)
        gp = np.exp(s[:, g] - gm)
        parts.append((gp / gp.sum(1, keepdims=True)) @ v[g])
        lses.append(gm[:, 0] + np.log(gp.sum(1)))
    P = np.stack(parts)[:, :, None, :]            # [n, T=3, H=1, Dv]
    L = np.stack(lses)[:, :, None]
    out, lse = R.ref_lse_merge(P, L, True)
    assert np.max(np.abs(out[:, 0] - full_out)) < 1e-12
    assert np.max(np.abs(lse[:, 0] - full_lse)) < 1e-12
    out2, lse2 = R.ref_lse_merge(P, L / math.log(2.0), False)
    assert np.max(np.abs(out2[:, 0] - full_out)) < 1e-12
    assert np.max(np.abs(lse2[:, 0] * math.log(2.0) - full_lse)) < 1e-12
    one, l1 = R.ref_lse_merge(P[:1], L[:1], True)
    assert np.max(np.abs(one - P[0])) == 0 and np.max(np.abs(l1 - L[0])) == 0
    e_out, e_lse = R.ref_lse_merge(np.ones((2, 3, 1, Dv)), np.full((2, 3, 1), -np.inf), True)
    assert np.all(e_out == 0) and np.all(np.isneginf(e_lse))


def check_lse_bases():
    q, rows = make_small_case(4, 2, 4, 2, (20, 33), 8)
    bt, nb = make_block_table(4, 2, 5)
    for cp in (1, 3):
        for rank in range(cp):
            pool = R.ref_build_pool(rows, bt, 8, cp, rank, nb)
            G = np.array([20, 33])
            sl = R.ref_local_len(G, cp, rank)
            oe, le = R.ref_mla_decode(q, pool, bt, sl, G, 2, cp, rank, 0.1, True)
            o2, l2 = R.ref_mla_decode(q, pool, bt, sl, G, 2, cp, rank, 0.1, False)
            assert np.array_equal(oe, o2)
            fin = np.isfinite(le)
            assert np.array_equal(fin, np.isfinite(l2))
            assert np.max(np.abs(l2[fin] * math.log(2.0) - le[fin]), initial=0) < 1e-12


def _shard_inputs(seed, B, H, q_len, G, bs, cp):
    q, rows = make_small_case(seed, B, H, q_len, G, bs)
    ppr = max(((n + cp - 1) // cp + bs - 1) // bs for n in G)
    bt, nb = make_block_table(seed, B, ppr)
    return q, rows, bt, nb


def check_merge_equals_unsharded():
    """Per-shard decode over each shard's pool, merged through the LSEs, equals the
    unsharded attention over global positions."""
    scale = 1.0 / math.sqrt(192.0)
    for seed, (B, H, q_len, G, bs, cp) in enumerate([
            (3, 4, 4, (1, 19, 70), 4, 2), (2, 3, 3, (2, 45), 8, 3),
            (2, 2, 2, (130, 9), 16, 8), (1, 2, 4, (33,), 4, 16)]):
        q, rows, bt, nb = _shard_inputs(seed, B, H, q_len, G, bs, cp)
        Ga = np.array(G)
        for base_e in (True, False):
            outs, lses = [], []
            for rank in range(cp):
                pool = R.ref_build_pool(rows, bt, bs, cp, rank, nb)
                sl = R.ref_local_len(Ga, cp, rank)
                o, l = R.ref_mla_decode(q, pool, bt, sl, Ga, q_len, cp, rank, scale, base_e)
                outs.append(o)
                lses.append(l)
            mo, ml = R.ref_lse_merge(np.stack(outs), np.stack(lses), base_e)
            go, gl = R.ref_attention_global(q, rows, Ga, q_len, scale)
            if not base_e:
                gl = gl / math.log(2.0)
            assert np.max(np.abs(mo - go)) < 1e-12, np.max(np.abs(mo - go))
            fin = np.isfinite(gl)
            assert np.array_equal(fin, np.isfinite(ml))
            assert np.max(np.abs(ml[fin] - gl[fin]), initial=0) < 1e-12


def check_pool_vs_global_formulation():
    scale = 0.07
    q, rows, bt, nb = _shard_inputs(9, 2, 3, 3, (26, 61), 4, 4)
    Ga = np.array([26, 61])
    for rank in range(4):
        pool = R.ref_build_pool(rows, bt, 4, 4, rank, nb)
        sl = R.ref_local_len(Ga, 4, rank)
        a = R.ref_mla_decode(q, pool, bt, sl, Ga, 3, 4, rank, scale, True)
        b = R.ref_mla_decode_global(q, rows, Ga, 3, 4, rank, scale, True)
        assert np.max(np.abs(a[0] - b[0])) < 1e-12
        assert np.array_equal(a[1], b[1])


def check_flattened_equals_native():
    """Legacy path: B*q_len single-token rows, block table repeated per row, each row's
    own local length as its seq_len and a very long global length, so that only
    seq_lens bounds it.  Must equal the native q_len-block result."""
    scale = 0.05
    B, H, q_len, G, bs, cp = 2, 3, 3, (29, 44), 4, 3
    q, rows, bt, nb = _shard_inputs(21, B, H, q_len, G, bs, cp)
    Ga = np.array(G)
    for rank in range(cp):
        pool = R.ref_build_pool(rows, bt, bs, cp, rank, nb)
        sl = R.ref_local_len(Ga, cp, rank)
        nat = R.ref_mla_decode(q, pool, bt, sl, Ga, q_len, cp, rank, scale, True)
        per_row = R.ref_local_len(R.ref_row_global_prefix(Ga, q_len).reshape(-1), cp, rank)
        qf = q.reshape(B * q_len, 1, H, -1)
        btf = np.repeat(bt, q_len, axis=0)
        huge = np.full(B * q_len, 1 << 40)
        flat = R.ref_mla_decode(qf, pool, btf, per_row, huge, 1, cp, rank, scale, True)
        assert np.max(np.abs(nat[0] - flat[0])) < 1e-12
        assert np.array_equal(nat[1], flat[1])


def check_end_aligned_mask_differs():
    """An end-aligned local mask (local_len - (q_len-1-i)) attends to the wrong keys on
    round-robin shards for q_len > 1 (the review on the "vLLM PR #48180" page); the
    oracle must not coincide with it."""
    scale = 0.1
    B, H, q_len, G, bs, cp = 1, 2, 4, (23,), 4, 4
    q, rows, bt, nb = _shard_inputs(31, B, H, q_len, G, bs, cp)
    Ga = np.array(G)
    differs = False
    for rank in range(cp):
        pool = R.ref_build_pool(rows, bt, bs, cp, rank, nb)
        sl = R.ref_local_len(Ga, cp, rank)
        o, _ = R.ref_mla_decode(q, pool, bt, sl, Ga, q_len, cp, rank, scale, True)
        for i in range(q_len):
            Lw = max(0, int(sl[0]) - (q_len - 1 - i))
            if Lw == 0:
                continue
            keys = R.ref_gather_pages(pool, bt[0], Lw)
            s = scale * (q[0, i] @ keys.T)
            p = np.exp(s - s.max(1, keepdims=True))
            ow = (p / p.sum(1, keepdims=True)) @ keys[:, :512]
            if np.max(np.abs(ow - o[i])) > 1e-6:
                differs = True
    assert differs


def check_abs_weighted_closed_form():
    """With non-negative V the error scale sum_l p_l |V_l| is the output itself."""
    q, rows = make_small_case(41, 2, 3, 2, (40, 77), 8)
    rows = [np.abs(r) for r in rows]
    G = np.array([40, 77])
    for cp, rank in ((1, 0), (3, 2)):
        o, _ = R.ref_mla_decode_global(q, rows, G, 2, cp, rank, 0.1, True)
        a = R.ref_abs_weighted(q, rows, G, 2, cp, rank, 0.1)
        assert np.max(np.abs(o - a)) < 1e-12


def _sdpa_unmasked(q_np, rows, G, scale):
    """torch float64 SDPA with no mask (every query row sees all G[b] keys), MQA
    broadcast over heads; returns (out, lse) rows ordered (b, i)."""
    outs, lses = [], []
    B, q_len, H, D = q_np.shape
    for b in range(B):
        K = torch.from_numpy(np.asarray(rows[b][:G[b]], dtype=np.float64))
        Qh = torch.from_numpy(np.asarray(q_np[b], dtype=np.float64)).permute(1, 0, 2)[None]
        Kh = K[None, None].expand(1, H, G[b], D)
        Vh = K[None, None, :, :512].expand(1, H, G[b], 512)
        o = torch.nn.functional.scaled_dot_product_attention(Qh, Kh, Vh, scale=scale)
        lse = torch.logsumexp((Qh @ Kh.transpose(-1, -2)) * scale, dim=-1)
        outs.append(o[0].permute(1, 0, 2).numpy())
        lses.append(lse[0].permute(1, 0).numpy())
    return np.concatenate(outs, 0), np.concatenate(lses, 0)


def check_noncausal_vs_sdpa():
    """A non-causal block (DSpark draft): every row sees the request's whole context.
    With one shard that is unmasked attention (library SDPA, float64), and each row
    equals an ordinary single-token decode of that row's query."""
    scale = 1.0 / math.sqrt(192.0)
    for seed, (B, H, q_len, G, bs) in enumerate([(2, 4, 3, (37, 130), 16),
                                                 (3, 2, 4, (1, 64, 65), 8)]):
        q, rows = make_small_case(100 + seed, B, H, q_len, G, bs)
        ppr = max((n + bs - 1) // bs for n in G)
        bt, nb = make_block_table(100 + seed, B, ppr)
        pool = R.ref_build_pool(rows, bt, bs, 1, 0, nb)
        Ga = np.array(G)
        out, lse = R.ref_mla_decode(q, pool, bt, Ga, None, q_len, 1, 0, scale, True,
                                    causal=False)
        ro, rl = _sdpa_unmasked(q, rows, list(G), scale)
        assert np.max(np.abs(out - ro)) < 1e-12, np.max(np.abs(out - ro))
        assert np.max(np.abs(lse - rl)) < 1e-12
        for i in range(q_len):
            o1, l1 = R.ref_mla_decode(q[:, i:i + 1], pool, bt, Ga, None, 1, 1, 0, scale, True)
            assert np.array_equal(o1, out[i::q_len]) and np.array_equal(l1, lse[i::q_len])


def check_noncausal_merge_equals_unsharded():
    """Non-causal shards (each row reads the shard's whole local sequence, seq_lens),
    merged through their LSEs, equal unmasked attention over the global sequence."""
    scale = 0.09
    for seed, (B, H, q_len, G, bs, cp, il) in enumerate([
            (2, 3, 3, (29, 50), 4, 3, 1), (2, 2, 4, (7, 66), 8, 2, 4), (1, 2, 2, (40,), 4, 8, 1)]):
        q, rows, bt, nb = _shard_inputs(200 + seed, B, H, q_len, G, bs, cp)
        Ga = np.array(G)
        outs, lses = [], []
        for rank in range(cp):
            pool = R.ref_build_pool(rows, bt, bs, cp, rank, nb, il)
            sl = R.ref_local_len(Ga, cp, rank, il)
            o, l = R.ref_mla_decode(q, pool, bt, sl, None, q_len, cp, rank, scale, True,
                                    interleave=il, causal=False)
            outs.append(o)
            lses.append(l)
            g = R.ref_mla_decode_global(q, rows, Ga, q_len, cp, rank, scale, True,
                                        interleave=il, causal=False)
            assert np.max(np.abs(o - g[0])) < 1e-12 and np.array_equal(l, g[1])
        mo, ml = R.ref_lse_merge(np.stack(outs), np.stack(lses), True)
        ro, rl = _sdpa_unmasked(q, rows, list(G), scale)
        assert np.max(np.abs(mo - ro)) < 1e-12, np.max(np.abs(mo - ro))
        assert np.max(np.abs(ml - rl)) < 1e-12
        go, gl = R.ref_attention_global(q, rows, Ga, q_len, scale, causal=False)
        assert np.max(np.abs(go - ro)) < 1e-12 and np.max(np.abs(gl - rl)) < 1e-12


def check_interleave_merge_equals_unsharded():
    """Causal shards under round-robin segments of ``interleave`` positions (pools laid
    out by the slot mapping with the same interleave), merged, equal causal attention
    over the unsharded sequence (library SDPA with a position mask)."""
    scale = 1.0 / math.sqrt(192.0)
    for seed, (B, H, q_len, G, bs, cp, il) in enumerate([
            (2, 3, 3, (29, 70), 4, 2, 2), (2, 2, 4, (9, 100), 8, 3, 4),
            (1, 2, 2, (66,), 6, 2, 3), (2, 2, 1, (5, 48), 16, 4, 16)]):
        q, rows, bt, nb = _shard_inputs(300 + seed, B, H, q_len, G, bs, cp)
        Ga = np.array(G)
        outs, lses = [], []
        for rank in range(cp):
            pool = R.ref_build_pool(rows, bt, bs, cp, rank, nb, il)
            sl = R.ref_local_len(Ga, cp, rank, il)
            o, l = R.ref_mla_decode(q, pool, bt, sl, Ga, q_len, cp, rank, scale, True,
                                    interleave=il)
            outs.append(o)
            lses.append(l)
            g = R.ref_mla_decode_global(q, rows, Ga, q_len, cp, rank, scale, True,
                                        interleave=il)
            assert np.max(np.abs(o - g[0])) < 1e-12 and np.array_equal(l, g[1])
        mo, ml = R.ref_lse_merge(np.stack(outs), np.stack(lses), True)
        ro, rl = _sdpa_reference(q, rows, list(G), q_len, scale)
        assert np.max(np.abs(mo - ro)) < 1e-12, np.max(np.abs(mo - ro))
        assert np.max(np.abs(ml - rl)) < 1e-12


def check_owned_positions():
    """The positions a shard holds, enumerated, number ref_local_len's closed form; the
    shards partition the sequence; and the k-th held position is the shard's local
    position k: the slot mapping puts it at page block_table[k // bs], offset k % bs."""
    rng = np.random.default_rng(8)
    for cp, il, bs in [(1, 1, 4), (2, 1, 4), (3, 2, 4), (4, 4, 8), (8, 1, 16), (2, 3, 6)]:
        nvb = 4
        bt = rng.permutation(40)[:nvb].reshape(1, nvb)
        G = nvb * bs * cp
        seen = np.zeros(G, dtype=int)
        for rank in range(cp):
            own = R.ref_owned_positions(G, cp, rank, il)
            seen[own] += 1
            for Gp in range(0, G + 1, 3):
                assert len(R.ref_owned_positions(Gp, cp, rank, il)) == \
                    int(R.ref_local_len(Gp, cp, rank, il))
            slots = R.ref_cp_local_slot(own.reshape(1, -1), bt, bs, cp, rank, il)[0]
            k = np.arange(own.size)
            assert np.array_equal(slots, bt[0, k // bs] * bs + k % bs), (cp, il, bs, rank)
        assert np.all(seen == 1)


def check_scatter_then_decode():
    """New KV rows scattered into each shard's pool through the slot mapping: context in
    one call, then a draft block whose rejected tail (negative positions) is skipped.
    Every slot another shard owns stays untouched (NaN), and decoding the pools gives the
    global-position formulation over the accepted rows."""
    scale = 0.08
    bs, cp, il = 4, 2, 2
    B, H, q_len = 2, 2, 1
    G = (22, 37)
    q, rows = make_small_case(400, B, H, q_len, G, bs)
    ppr = max(((n + cp - 1) // cp + bs - 1) // bs for n in G) + 1
    bt, nb = make_block_table(400, B, ppr)
    acc = (18, 33)                                   # accepted length; the rest rejected
    for rank in range(cp):
        pool = np.full((nb, bs, 576), np.nan)
        Nc = max(acc) - 4
        pos_c = np.full((B, Nc), -1, dtype=np.int64)
        kv_c = np.zeros((B, Nc, 576))
        for b in range(B):
            n = acc[b] - 4
            pos_c[b, :n] = np.arange(n)
            kv_c[b, :n] = rows[b][:n]
        pool = R.ref_scatter_kv(pool, pos_c, kv_c, bt, bs, cp, rank, il)
        pos_d = np.full((B, 8), -1, dtype=np.int64)
        kv_d = np.zeros((B, 8, 576))
        for b in range(B):
            base = acc[b] - 4
            pos_d[b, :4] = base + np.arange(4)                 # accepted draft rows
            kv_d[b] = rows[b][base:base + 8]                   # rejected rows stay -1
        pool = R.ref_scatter_kv(pool, pos_d, kv_d, bt, bs, cp, rank, il)
        want = R.ref_build_pool([r[:a] for r, a in zip(rows, acc)], bt, bs, cp, rank, nb, il)
        assert np.array_equal(np.isnan(pool), np.isnan(want))
        fin = ~np.isnan(want)
        assert np.array_equal(pool[fin], want[fin])
        Ga = np.array(acc)
        sl = R.ref_local_len(Ga, cp, rank, il)
        a = R.ref_mla_decode(q, pool, bt, sl, Ga, q_len, cp, rank, scale, True, interleave=il)
        g = R.ref_mla_decode_global(q, rows, Ga, q_len, cp, rank, scale, True, interleave=il)
        assert np.max(np.abs(a[0] - g[0])) < 1e-12 and np.array_equal(a[1], g[1])


ALL_CHECKS = [check_noncausal_vs_sdpa, check_noncausal_merge_equals_unsharded,
              check_interleave_merge_equals_unsharded, check_owned_positions,
              check_scatter_then_decode,
              check_slot_golden, check_local_len_golden, check_local_len_bruteforce,
              check_row_prefix_positions, check_slot_bruteforce, check_decode_vs_sdpa,
              check_decode_bruteforce_tiny, check_merge_closed_form, check_lse_bases,
              check_merge_equals_unsharded, check_pool_vs_global_formulation,
              check_flattened_equals_native, check_end_aligned_mask_differs,
              check_abs_weighted_closed_form]
