"""Property checks for a balanced plan, written from the pages' invariants.

These checks do not recompute the plan; they verify what any plan produced by
the rule must satisfy:

* every rank receives exactly S*K routes (MoonshotAI/MoonEP README, item 1);
* dst is a bijection from routes onto valid, non-padding rows, and its sign
  marks a later route of a token that lands on a rank already holding an
  earlier route of that token (MoonEP Public API Visual Guide,
  Buffer.dispatch(...) and Buffer.combine(...): positive/negative encoding);
* at most B prefetch slots per rank, all holding experts of a single remote
  home group (README, "How to set B");
* cu_seqlens holds padded end offsets, monotone and aligned to token_padding,
  and unused slots have an empty segment (Visual Guide, Buffer(...)
  token_padding; vllm MoonEP MoonEPExpertWeightLayout);
* home segments hold only their own expert, slot segments only the slot's
  expert, and rows inside a segment follow (source rank, s, k) order;
* each rank keeps a prefix of its home-group routes ordered by
  (expert, source rank, s, k).
"""
from __future__ import annotations

import numpy as np


def decode(dst: np.ndarray) -> np.ndarray:
    d = dst.astype(np.int64)
    return np.where(d >= 0, d, -d - 1)


def check_plan(cfg: dict, topk: np.ndarray, p: dict, max_records: int = 4096) -> dict:
    R, E, K, S, B, tp = (cfg[k] for k in ("R", "E", "K", "S", "B", "tp"))
    L, C, EB = E // R, S * K, E + B
    NvS = p["NvS"]
    ids = np.asarray(topk, np.int64).reshape(R, C)
    dst = np.asarray(p["dst"]).reshape(R, C)
    etc = np.asarray(p["experts_to_copy"]).reshape(R, B)
    cu = np.asarray(p["cu_seqlens"]).reshape(R, EB).astype(np.int64)
    zfr = np.asarray(p["zero_fill_ranges"]).reshape(R, EB, 2).astype(np.int64)
    g = decode(dst)
    j_of = g // NvS
    w_of = g % NvS

    assert g.min() >= 0 and g.max() < R * NvS
    # bijection onto distinct rows
    assert len(np.unique(g)) == R * C, "dst is not injective"
    # every rank receives exactly C routes
    assert np.all(np.bincount(j_of.reshape(-1), minlength=R) == C)

    # cu_seqlens: monotone, aligned, bounded; starts and valid counts
    starts = np.concatenate([np.zeros((R, 1), np.int64), cu[:, :-1]], axis=1)
    assert np.all(np.diff(cu, axis=1) >= 0)
    assert np.all(cu % tp == 0)
    assert np.all(cu[:, -1] <= NvS)
    n = zfr[:, :, 0] - starts
    assert np.all(n >= 0)
    assert np.all(zfr[:, :, 1] == cu)
    assert np.all((n + tp - 1) // tp * tp == cu - starts)

    # segment of every route; rows must lie in the valid part
    seg = np.full((R, C), -1, np.int64)
    for j in range(R):
        sel = j_of == j
        w = w_of[sel]
        x = np.searchsorted(cu[j], w, side="right")
        assert np.all(x < EB)
        assert np.all(w < zfr[j, x, 0]), "route lands on a padding row"
        seg[sel] = x
    # valid counts match the number of routes landing in each segment
    for j in range(R):
        cnt = np.bincount(seg[j_of == j], minlength=EB)
        assert np.array_equal(cnt, n[j])

    # slots: contiguous from 0, at most B, ascending ids, one remote group
    for j in range(R):
        used = etc[j][etc[j] >= 0]
        nu = len(used)
        assert np.all(etc[j][:nu] >= 0) and np.all(etc[j][nu:] == -1)
        assert np.all(np.diff(used) > 0)
        if nu:
            groups = np.unique(used // L)
            assert len(groups) == 1 and groups[0] != j
            assert nu <= min(B, L)
        for b in range(B):
            empty = n[j, E + b] == 0
            assert empty == (etc[j, b] < 0), "slot use and segment disagree"
        # non-home expert segments are empty
        for x in range(E):
            if x // L != j:
                assert n[j, x] == 0

    # content of each segment
    home_seg = seg < E
    assert np.all(seg[home_seg] == ids[home_seg])
    assert np.all(ids[home_seg] // L == j_of[home_seg])
    slot_e = etc[j_of[~home_seg], seg[~home_seg] - E]
    assert np.all(slot_e == ids[~home_seg])

    # Q order inside segments: rows contiguous and in route-id (r, s, k) order
    fg = g.reshape(-1)
    fs = (j_of * EB + seg).reshape(-1)
    rid = np.arange(R * C)
    o = np.lexsort((fg, fs))
    same = fs[o][1:] == fs[o][:-1]
    assert np.all(np.diff(fg[o])[same] == 1), "segment rows not contiguous"
    assert np.all(np.diff(rid[o])[same] > 0), "segment rows not in (r,s,k) order"

    # each rank keeps a prefix of Q_j in (expert, r, s, k) order
    for j in range(R):
        home = (ids // L) == j
        rr, ii = np.nonzero(home)
        key = np.lexsort((ii, rr, ids[rr, ii]))
        stays = (j_of[rr, ii] == j)[key]
        kept = int(stays.sum())
        assert np.all(stays[:kept]) and not np.any(stays[kept:]), "kept routes are not a prefix of Q_j"

    # duplicate sign rule
    jt = j_of.reshape(R * S, K)
    neg = (dst.reshape(R * S, K) < 0)
    for k in range(K):
        earlier = np.zeros(R * S, bool)
        for k2 in range(k):
            earlier |= jt[:, k2] == jt[:, k]
        assert np.array_equal(earlier, neg[:, k]), "dst sign disagrees with the duplicate rule"

    # statistics
    rs = np.asarray(p["remote_stats"]).reshape(R, 2)
    dc = np.asarray(p["dup_counts"]).reshape(R, 2)
    for j in range(R):
        on_j = j_of == j
        assert rs[j, 0] == int((on_j & ((ids // L) != j)).sum())
        assert rs[j, 1] == int((etc[j] >= 0).sum())
        assert dc[j, 0] == int((on_j & (dst < 0)).sum())
        prim_with_dup = 0
        for k in range(K):
            later = np.zeros(R * S, bool)
            for k2 in range(k + 1, K):
                later |= jt[:, k2] == j
            prim_with_dup += int(((jt[:, k] == j) & ~neg[:, k] & later).sum())
        assert dc[j, 1] == prim_with_dup

    # duplicate records (CSR by primary row)
    if "dup_groups" in p and p["dup_groups"] is not None:
        dg = np.asarray(p["dup_groups"]).reshape(R, NvS, 3)
        dl = np.asarray(p["dup_loffs"]).reshape(R, NvS)
        gdst = g.reshape(R * S, K)
        inv = np.full(R * NvS, -1, np.int64)
        inv[g.reshape(-1)] = np.arange(R * C)
        for j in range(R):
            ng, nd = dc[j, 1], dc[j, 0]
            recs = dg[j, :ng]
            assert np.all(np.diff(recs[:, 0]) > 0)
            assert np.array_equal(recs[:, 1], np.concatenate([[0], np.cumsum(recs[:, 2])[:-1]]).astype(recs.dtype)) if ng else True
            assert int(recs[:, 2].sum()) == nd
            for prow, start, count in recs[:max_records]:
                # the primary's token and its duplicates on rank j
                t, k = divmod(int(inv[j * NvS + prow]), K)
                assert not neg[t, k]
                want = [int(gdst[t, k2] - j * NvS) for k2 in range(k + 1, K) if jt[t, k2] == j]
                assert list(dl[j, start:start + count]) == want
    moved = int((j_of != (ids // L)).sum())
    G = np.bincount((ids // L).reshape(-1), minlength=R)
    return {"moved": moved, "lower_bound": int(np.maximum(G - C, 0).sum()), "G": G}
