"""FS-B cell selection by beam search over two causal forests: plain numpy,
float64.

TEST INFRASTRUCTURE ONLY: the tests call it; the product path never imports
it, and it imports nothing from the product.

"FreeSolo: Linear-time Sparse Attention with Zero-Shot Length Extrapolation"
(ai.info summary, "Methodology in Plain English", the FS-B paragraph;
paper.rainbus.top summary, 方法步骤详情 ⑤ and 技术新颖性): FS-B keeps every
cell (no pruning) and builds two balanced trees per head, one over the full
prefix and one over the cells whose largest key norm exceeds a threshold tau
(set once per model; an input here).  Every node stores a mean key, a radius
bounding its children, the largest cell norm beneath it and the earliest
position beneath it.  A beam of 16 nodes per level descends each tree, ranked
by a provable upper bound on the score of every cell beneath a node; the union
of both beams' cells is reranked by the log-sum-exp of the token logits of
each cell, and the top K cells are read.

Readings taken (the pages give no formulas):
  * cell score: the FS / FS-L score, u_c = q . kbar_c + lambda a_c erf(sigma
    (n - p_c) / s), p_c = c s + s / 2;
  * the trees are causal forests over the cells in position order: the leaves
    of a forest are its cells in order, a node covers an aligned run of 2^j
    consecutive leaves, and a query of block beta uses the maximal aligned
    runs that tile the forest's available prefix (the binary decomposition of
    its length), so no node mixes available and unavailable cells;
  * node summaries: mean key = the mean of the cells' mean keys; radius r =
    the largest distance from the node's mean key to a cell mean key beneath
    it, bounded recursively as max over children (|mean_child - mean| +
    r_child); largest norm a_max; earliest position = the node's first cell;
  * bound: u_c <= q . mean + |q| r + lambda a_max erf(sigma (n - p_first) / s)
    (Cauchy-Schwarz for the content term; erf increasing in the distance,
    which is largest at the earliest cell, and lambda, a_c >= 0);
  * beam descent: every node of the beam is replaced by its children (a leaf
    by itself) and the best `beam` by bound are kept (ties: lower first cell),
    until the beam holds only leaves;
  * rerank: LSE_c = log sum_{t in c} exp(q . k_t / sqrt(d)), top K by (LSE
    desc, c asc) over the union of both beams.
"""
from __future__ import annotations

import math

import numpy as np


def build_forest(cells, kbar, amax):
    """Levels of the forest over `cells` (cell ids in position order):
    levels[j] = dict(mean [m_j, d], radius [m_j], amax [m_j], first [m_j]) for
    the aligned runs of 2^j leaves (the last run may be partial)."""
    cells = np.asarray(cells, np.int64)
    levels = [dict(mean=kbar[cells].astype(np.float64), radius=np.zeros(len(cells)),
                   amax=amax[cells].astype(np.float64), first=cells.copy())]
    while len(levels[-1]["mean"]) > 1:
        prev = levels[-1]
        m = len(prev["mean"])
        nm = (m + 1) // 2
        mean = np.zeros((nm, kbar.shape[1]))
        radius = np.zeros(nm)
        am = np.zeros(nm)
        first = np.zeros(nm, np.int64)
        for i in range(nm):
            kids = [2 * i] + ([2 * i + 1] if 2 * i + 1 < m else [])
            # equal-size children except a partial last run: weight by leaves
            w = np.array([min(2 ** (len(levels) - 1), len(cells) - c * 2 ** (len(levels) - 1))
                          for c in kids], np.float64)
            mean[i] = (w[:, None] * prev["mean"][kids]).sum(0) / w.sum()
            radius[i] = max(np.linalg.norm(prev["mean"][c] - mean[i]) + prev["radius"][c]
                            for c in kids)
            am[i] = max(prev["amax"][c] for c in kids)
            first[i] = prev["first"][kids[0]]
        levels.append(dict(mean=mean, radius=radius, amax=am, first=first))
    return levels


def node_bound(q, lev, i, n, lam, sigma, s):
    """Upper bound on the score of every cell beneath node i of a level."""
    p_first = lev["first"][i] * s + 0.5 * s
    return (float(q @ lev["mean"][i]) + float(np.linalg.norm(q)) * lev["radius"][i]
            + lam * lev["amax"][i] * math.erf(sigma * (n - p_first) / s))


def roots(m):
    """(level, index) of the maximal aligned runs tiling leaves [0, m)."""
    out, start = [], 0
    for j in reversed(range(max(1, m).bit_length())):
        if m & (1 << j):
            out.append((j, start >> j))
            start += 1 << j
    return out


def beam_search(q, levels, m, n, lam, sigma, s, beam):
    """Cells (leaf positions in the forest) the beam ends on, and the smallest
    relative gap between the last kept and the first dropped bound over the
    levels (a near tie there can change the result)."""
    if m == 0:
        return [], math.inf
    cur = roots(m)
    gap = math.inf
    while any(j > 0 for j, _ in cur):
        nxt = []
        for j, i in cur:
            nxt += [(j, i)] if j == 0 else [(j - 1, 2 * i), (j - 1, 2 * i + 1)]
        scored = sorted(((-node_bound(q, levels[j], i, n, lam, sigma, s), i << j, j, i)
                         for j, i in nxt))
        if len(scored) > beam:
            a, b = -scored[beam - 1][0], -scored[beam][0]
            gap = min(gap, abs(a - b) / max(abs(a), abs(b), 1e-300))
        cur = [(j, i) for _, _, j, i in scored[:beam]]
    return [i for _, i in cur], gap


def token_lse(q, k, c, s):
    logits = k[c * s:(c + 1) * s] @ q / math.sqrt(q.shape[0])
    mx = logits.max()
    return float(mx + math.log(np.exp(logits - mx).sum()))


def fsb_select_row(q, k, kbar, amax, n, lam, sigma, tau, s=32, Bq=128, K=4, beam=16):
    """Selected cells of query n (ranked by LSE, at most K) and the deciding
    gaps (beam boundary; K-th vs (K+1)-th LSE).  q [d]; k [N, d] unrotated
    keys; kbar [C, d], amax [C] of the same keys."""
    q = np.asarray(q, np.float64)
    A = (n // Bq) * Bq // s
    full = np.arange(A)
    high = np.nonzero(amax[:A] > tau)[0]
    cand, gap = set(), math.inf
    for cells in (full, high):
        if len(cells) == 0:
            continue
        lv = build_forest(cells, kbar, amax)
        leaves, g = beam_search(q, lv, len(cells), n, lam, sigma, s, beam)
        gap = min(gap, g)
        cand.update(int(cells[x]) for x in leaves)
    ranked = sorted((-token_lse(q, k, c, s), c) for c in cand)
    sel = [c for _, c in ranked[:K]]
    lse_gap = math.inf
    if len(ranked) > K:
        a, b = -ranked[K - 1][0], -ranked[K][0]
        lse_gap = abs(a - b) / max(abs(a), abs(b), 1e-300)
    return sel, gap, lse_gap


def fsb_select(q, k, kbar, amax, lam, sigma, tau, rows, s=32, Bq=128, K=4, beam=16):
    """fsb_select_row for every row in `rows` of one head: sel [R, K] (-1
    padded), beam gaps [R], rerank gaps [R]."""
    sel = np.full((len(rows), K), -1, np.int32)
    gaps = np.zeros(len(rows))
    lgaps = np.zeros(len(rows))
    for i, n in enumerate(rows):
        c, g, lg = fsb_select_row(q[n], k, kbar, amax, int(n), lam, sigma, tau, s, Bq, K, beam)
        sel[i, :len(c)] = c
        gaps[i], lgaps[i] = g, lg
    return sel, gaps, lgaps
