"""An independent, sort-based restatement of the balanced plan rule.

Written from the rule as stated (and from the pages' contracts), vectorised
with numpy sorts and prefix sums instead of the oracle's loops, so that a
mistake in either one shows up as a difference between the two:

1. P_e = the routes of expert e in (source rank, s, k) order -- a stable sort
   of the route ids by expert; Q_j = P_{jL} .. P_{jL+L-1}, G_j = |Q_j|.
2. Chain: while some rank holds fewer than C = S*K routes, the lowest such
   rank takes C - rem from the lowest rank holding more than C; each rank
   receives at most once, a donor keeps a prefix of Q_j and its pieces are
   consecutive runs after that prefix, in recording order.
3. Slots: on a receiver, the experts with at least one route in its run, in
   ascending id, take slots 0, 1, ...
4. Segments x = e (home expert, kept routes) and x = E + b (slot b), padded
   to token_padding; cu_seqlens are inclusive padded ends; zero-fill ranges
   cover each segment's padding; rows inside a segment follow Q order.
5. dst = j*NvS + row, encoded -(g+1) when an earlier route of the same token
   lands on the same rank; NvS = roundup(C + (L+B)(tp-1), tp).
("MoonshotAI/MoonEP" README items 1-2 and "How to set B"; "MoonEP Public API
Visual Guide", Buffer(...), Buffer.dispatch(...), MoonEPCommPlan.)
"""
from __future__ import annotations

import numpy as np


def restate_plan(R, E, K, S, B, tp, topk):
    """Returns (status, plan dict) with the oracle's field names; status -4
    when a receiver would need more than B slots."""
    L, C = E // R, S * K
    N = R * C
    ids = np.asarray(topk, np.int64).reshape(-1)          # route id = r*C + s*K + k
    NvS = -(-(C + (L + B) * (tp - 1)) // tp) * tp
    EB = E + B

    # 1. Q order
    T = np.bincount(ids, minlength=E)
    Pstart = np.concatenate([[0], np.cumsum(T)])           # P_e inside the (e, r, s, k) order
    home_first = (np.arange(E) // L) * L
    qoff = Pstart[:E] - Pstart[home_first]                 # offset of P_e inside Q_home(e)
    G = T.reshape(R, L).sum(axis=1)
    order = np.argsort(ids, kind="stable")
    pos_in_P = np.empty(N, np.int64)
    pos_in_P[order] = np.arange(N) - Pstart[ids[order]]
    q = qoff[ids] + pos_in_P                               # Q position of every route

    # 2. chain
    rem = G.astype(np.int64).copy()
    donated = np.zeros(R, np.int64)
    pieces = []                                            # (donor, receiver, length)
    while (rem < C).any():
        s_ = int(np.nonzero(rem < C)[0][0])
        l_ = int(np.nonzero(rem > C)[0][0])
        d = int(C - rem[s_])
        pieces.append((l_, s_, d))
        rem[l_] -= d
        donated[l_] += d
        rem[s_] = C
    keep = G - donated
    start = {}                                             # piece -> first Q position of its run
    run_end = keep.copy()
    for i, (l_, s_, d) in enumerate(pieces):
        start[i] = int(run_end[l_])
        run_end[l_] += d

    # 3. slots, 4. segment sizes
    n = np.zeros((R, EB), np.int64)
    etc = np.full((R, B), -1, np.int64)
    slot_of = {}                                           # (receiver, expert) -> slot
    recv_piece = {}
    for e in range(E):
        j = e // L
        n[j, e] = min(max(keep[j] - qoff[e], 0), T[e])
    for i, (l_, j, d) in enumerate(pieces):
        recv_piece[j] = i
        a = start[i]
        b = 0
        for e in range(l_ * L, (l_ + 1) * L):
            lo, hi = max(a, qoff[e]), min(a + d, qoff[e] + T[e])
            if T[e] > 0 and hi > lo:
                if b >= B:
                    return -4, None
                etc[j, b] = e
                slot_of[(j, e)] = b
                n[j, E + b] = hi - lo
                b += 1
    padded = -(-n // tp) * tp
    cu = np.cumsum(padded, axis=1)
    seg_start = cu - padded
    zfr = np.stack([seg_start + n, cu], axis=-1)

    # 5. rows and dst
    e_r = ids
    l_r = e_r // L
    j_r = np.where(q < keep[l_r], l_r, -1)
    row = np.where(j_r >= 0, seg_start[np.maximum(j_r, 0), e_r] + q - qoff[e_r], 0)
    for i, (l_, j, d) in enumerate(pieces):
        a = start[i]
        sel = (l_r == l_) & (q >= a) & (q < a + d)
        es = e_r[sel]
        b = np.array([slot_of[(j, int(e))] for e in es], np.int64)
        j_r[sel] = j
        row[sel] = seg_start[j, E + b] + q[sel] - np.maximum(a, qoff[es])
    g = j_r * NvS + row
    jt = j_r.reshape(R * S, K)
    primary = np.ones((R * S, K), bool)
    for k in range(1, K):
        for k2 in range(k):
            primary[:, k] &= jt[:, k2] != jt[:, k]
    has_dup = np.zeros((R * S, K), bool)
    for k in range(K):
        for k2 in range(k + 1, K):
            has_dup[:, k] |= jt[:, k2] == jt[:, k]
    gt = g.reshape(R * S, K)
    dst = np.where(primary, gt, -(gt + 1)).reshape(R, C)

    remote = np.zeros((R, 2), np.int64)
    for j in range(R):
        if j in recv_piece:
            remote[j, 0] = pieces[recv_piece[j]][2]
        remote[j, 1] = int((etc[j] >= 0).sum())
    dup = np.zeros((R, 2), np.int64)
    np.add.at(dup[:, 0], jt[~primary], 1)
    np.add.at(dup[:, 1], jt[primary & has_dup], 1)
    out = {"dst": dst.astype(np.int32), "experts_to_copy": etc.astype(np.int32),
           "cu_seqlens": cu.astype(np.int32), "zero_fill_ranges": zfr.astype(np.int32),
           "remote_stats": remote.astype(np.int32), "dup_counts": dup.astype(np.int32),
           "NvS": NvS}
    return 0, out
