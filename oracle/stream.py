"""Streaming FS-L decoding with a bounded state: plain numpy, float64.

TEST INFRASTRUCTURE ONLY: the tests call it; the product path never imports
it, and it imports nothing from the product.

"FreeSolo: Linear-time Sparse Attention with Zero-Shot Length Extrapolation"
(ai.info summary, "Methodology in Plain English": FS-L keeps a bounded pool
of at most 72 cells, 8 recent plus the 64 with the largest key norm, which
updates only at query-block boundaries, so the streaming cache is small;
paper.rainbus.top summary, 核心方法: FS-L has linear cost and a bounded state,
and 实验结果: the FS-L attention buffer stays constant from 4k to 256k).

One token at a time, the decoder keeps only:
- the last w tokens (key, value, position) for the window branch;
- the open cell's rows;
- closed cells not yet available (they become available at the next block
  start: at most Bq/s of them);
- the W most recent available cells and the running top-P of the older ones,
  each with its summary (mean key, largest key norm) and its raw rows.

A cell that leaves the recent set enters the running top-P by (a_c desc,
c asc), or is dropped with its rows.  The top-P threshold only rises, since
the kept set can only admit new cells, so a dropped cell is never needed
again.  That is what bounds the state.  Each query then scores the pool
(content term plus the norm-weighted erf bias), keeps the top K (u desc,
c asc), reads the selected cells' raw rows (NoPE softmax, then RMSNorm) and
the window (RoPE softmax), and mixes the two, as the definition-form forward
does from the whole history.
"""
from __future__ import annotations

import math
from collections import deque

import numpy as np


def _rope(x, pos, base):
    d = x.shape[-1]
    h = d // 2
    theta = base ** (-2.0 * np.arange(h) / d)
    ang = pos * theta
    c, s = np.cos(ang), np.sin(ang)
    return np.concatenate([x[:h] * c - x[h:] * s, x[:h] * s + x[h:] * c])


def decode_stream(q, k, v, lam, sigma, mix, params):
    """Outputs of every row of one head slice (q, k, v [N, d] float values),
    decoded token by token from the bounded state.  Returns (out [N, d],
    sel [N, K] int32 with -1 padding, the largest number of token rows the
    state held at any step, and that bound)."""
    w, s, K, P, W, Bq = (params[x] for x in ("w", "s", "K", "P", "W", "Bq"))
    base, eps = params["rope_base"], params["rms_eps"]
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    N, d = q.shape
    scale = 1.0 / math.sqrt(d)
    window = deque()          # (position, rotated key, value), at most w
    open_rows = []            # (key, value) of the cell being filled
    pending = []              # closed cells not yet available
    recent = []               # ids of the W newest available cells
    top = []                  # running top-P older cells: (a, c) in rank order
    cells = {}                # id -> (kbar, a, keys [s, d], values [s, d])
    out = np.zeros((N, d))
    sel = np.full((N, K), -1, np.int32)
    held_max = 0
    bound = w + s + (Bq // s + W + P) * s
    for t in range(N):
        if t % Bq == 0:  # block start: the cells closed so far become available
            recent.extend(pending)
            pending = []
            while len(recent) > W:  # the oldest recent cell joins the older cells
                c = recent.pop(0)
                a = cells[c][1]
                pos = 0
                while pos < len(top) and (top[pos][0] > a or (top[pos][0] == a and top[pos][1] < c)):
                    pos += 1
                top.insert(pos, (a, c))
                if len(top) > P:
                    _, dropped = top.pop()
                    del cells[dropped]
        window.append((t, _rope(k[t], float(t), base), v[t]))
        if len(window) > w:
            window.popleft()
        open_rows.append((k[t], v[t]))
        held = (len(window) + len(open_rows)
                + s * (len(pending) + len(recent) + len(top)))
        held_max = max(held_max, held)
        # long branch: score the pool, keep the top K, read their raw rows
        pool = recent + [c for _, c in top]
        scored = []
        for c in pool:
            kbar_c, a_c = cells[c][0], cells[c][1]
            p_c = c * s + 0.5 * s
            u = float(q[t] @ kbar_c) + lam * a_c * math.erf(sigma * (t - p_c) / s)
            scored.append((-u, c))
        scored.sort()
        chosen = [c for _, c in scored[:K]]
        sel[t, :len(chosen)] = chosen
        o_long = np.zeros(d)
        if chosen:
            keys = np.concatenate([cells[c][2] for c in chosen])
            vals = np.concatenate([cells[c][3] for c in chosen])
            logit = keys @ q[t] * scale
            p = np.exp(logit - logit.max())
            o = (p @ vals) / p.sum()
            o_long = o / math.sqrt(float(o @ o) / d + eps)
        # window branch
        qr = _rope(q[t], float(t), base)
        kw = np.stack([x[1] for x in window])
        vw = np.stack([x[2] for x in window])
        logit = kw @ qr * scale
        p = np.exp(logit - logit.max())
        o_win = (p @ vw) / p.sum()
        out[t] = o_win + mix * o_long
        # the token closes its cell: summary, then available at the next block start
        if (t + 1) % s == 0:
            ks = np.stack([r[0] for r in open_rows])
            vs = np.stack([r[1] for r in open_rows])
            c = t // s
            cells[c] = (ks.mean(axis=0), float(np.sqrt((ks * ks).sum(axis=1)).max()), ks, vs)
            pending.append(c)
            open_rows = []
    return out, sel, held_max, bound
