"""Workloads that need the oracle to build (planted ties, needles).

Both are built on the CPU from the seeded generator plus the oracle's FP64
scores; the CUDA path never contributes to an input or an expected value.
"""

from __future__ import annotations

import numpy as np

from sparse_attention_kv_qsa_gb300 import workloads as w


def _desc_order(S_row: np.ndarray) -> np.ndarray:
    return np.lexsort((np.arange(S_row.shape[0]), -S_row))


def tiny_with_ties(o) -> w.Workload:
    """nq=8, 1,024 blocks, k=64, N(0,1), with 4 bit-identical blocks per
    query straddling the k boundary.

    For query i (in order): the source is the block at sorted position k-1
    (1-based), else k-2 or k, so the 4-block group occupies positions
    p..p+3 around the boundary (two in and two out at p = k-1). Its key is
    copied into three other blocks -- two with lower ids, one with a higher
    id, drawn from the seeded tie stream -- chosen among blocks that no
    group uses and that rank below the boundary for this query and for
    every query planted before it; the source must also score below every
    earlier query's group, so earlier groups keep their positions. After the
    last query every group is re-verified against the oracle.
    """
    W = w.tiny()
    k, n = W.k, W.active
    kb = W.kblk.copy()
    u = w.uniform(w.seed_for(0), w.STREAM_TIES, 100000)
    ui = 0
    used: set[int] = set()
    groups = []
    S = o.scores(W.q, kb, n)
    for i in range(W.nq):
        order = _desc_order(S[i])
        source = None
        for pos1 in (k - 1, k - 2, k):
            cand = int(order[pos1 - 1])
            if cand in used:
                continue
            if all(S[j][cand] < S[j][g[0]] for j, g in enumerate(groups)):
                source = cand
                break
        assert source is not None, f"no admissible tie source for query {i}"
        rank = np.empty(n, dtype=np.int64)
        rank[order] = np.arange(n)
        ok = [b for b in range(n)
              if b not in used and b != source and rank[b] > k + 8
              and all(S[j][b] < S[j][g[0]] for j, g in enumerate(groups))]
        lower = [b for b in ok if b < source]
        higher = [b for b in ok if b > source]
        assert len(lower) >= 2 and len(higher) >= 1
        picks = []
        for pool, cnt in ((lower, 2), (higher, 1)):
            pool = list(pool)
            for _ in range(cnt):
                j = int(u[ui] * len(pool))
                ui += 1
                picks.append(pool.pop(j))
        for b in picks:
            kb[b] = kb[source]
        group = sorted([source] + picks)
        used.update(group)
        groups.append(group)
        S = o.scores(W.q, kb, n)
    for i, g in enumerate(groups):
        vals = S[i][g]
        assert np.all(vals == vals[0]), "tie group not bit-identical"
        order = _desc_order(S[i])
        pos = sorted(int(np.nonzero(order == b)[0][0]) for b in g)
        assert pos == list(range(pos[0], pos[0] + 4)), "tie group not contiguous"
        assert pos[0] <= k - 1 < pos[3], "tie group does not straddle the boundary"
    W.kblk = kb
    W.name = "tiny_4k_nq8_k64_ties"
    W.meta["tie_groups"] = groups
    return W


def long_with_needles(o) -> w.Workload:
    """131,072 cells (32,768 blocks), nq=256, k=256: for each query, 16
    needle blocks get their key's projection on the query's unit head-sum
    direction s^ raised to |c| + 6 (c the old projection), so each needle
    scores |sum_h q_h| * (|c| + 6), at least 6 standard deviations of the
    query's score distribution. The oracle confirms every needle is
    selected."""
    W = w.long()
    kb = W.kblk.copy()
    qs = W.q.astype(np.float64).sum(axis=1)
    shat = qs / np.linalg.norm(qs, axis=1, keepdims=True)
    for i in range(W.nq):
        for b in W.meta["needles"][i]:
            row = kb[b].astype(np.float64)
            c = float(shat[i] @ row)
            kb[b] = (row + (abs(c) + 6.0 - c) * shat[i]).astype(np.float32)
    W.kblk = kb
    return W
