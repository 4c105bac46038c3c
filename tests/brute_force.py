"""Independent dense fp64 restatement of the FS / FS-L forward for tiny N.

Used only to pin the oracle.  It shares nothing with ``oracle/fs_oracle.c``:
instead of sorting and looping it builds dense masks -- an [N, C] availability
mask, pool membership by counting how many older cells outrank each cell, the
top-K by counting how many pool cells outscore each cell, an [N, N] token
mask -- and runs masked dense softmax attention.  RoPE is applied as a complex
multiplication of the pairs (x_i + i*x_{i+d/2}) by exp(i*pos*theta_i).

Method as read from the FreeSolo pages ("FreeSolo: Linear-time Sparse
Attention with Zero-Shot Length Extrapolation": paper.rainbus.top summary,
核心方法 and 方法步骤详情 ②-⑥; ai.info summary, "Methodology in Plain English").
"""
from __future__ import annotations

import numpy as np
from scipy.special import erf


def rope_complex(x, pos, base):
    N, d = x.shape
    h = d // 2
    theta = base ** (-np.arange(h) * 2.0 / d)
    z = (x[:, :h] + 1j * x[:, h:]) * np.exp(1j * np.outer(pos, theta))
    return np.concatenate([z.real, z.imag], axis=1)


def masked_softmax_attention(logits, mask, v):
    logits = np.where(mask, logits, -np.inf)
    has = mask.any(axis=1)
    mx = np.where(has, logits.max(axis=1, initial=-np.inf), 0.0)
    p = np.where(mask, np.exp(logits - mx[:, None]), 0.0)
    den = p.sum(axis=1)
    out = (p @ v) / np.where(has, den, 1.0)[:, None]
    return out, has


def brute_forward(q, k, v, lam, sigma, mix, w=512, s=32, K=4, P=64, W=8, Bq=128,
                  rope_base=10000.0, rms_eps=1e-6, mode=0, pos_offset=0.0, **_):
    """One head.  q, k, v: [N, d] float64.  Returns dict of dense results."""
    q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    N, d = q.shape
    C = N // s
    n = np.arange(N)
    c = np.arange(C)

    cell_k = k.reshape(C, s, d)
    kbar = cell_k.mean(axis=1)
    amax = np.linalg.norm(cell_k, axis=2).max(axis=1)

    b0 = (n // Bq) * Bq
    avail = (c[None, :] + 1) * s <= b0[:, None]                      # [N, C]
    n_avail = avail.sum(axis=1)
    if mode == 0:
        recent = avail & (c[None, :] >= (n_avail - W)[:, None])
        older = avail & ~recent
        # outranks[c2, c1]: c2 ranks above c1 by (a desc, c asc)
        outranks = (amax[:, None] > amax[None, :]) | (
            (amax[:, None] == amax[None, :]) & (c[:, None] < c[None, :]))
        rank = older.astype(np.int64) @ outranks.astype(np.int64)    # [N, C]
        pool = recent | (older & (rank < P))
    else:
        pool = avail

    p_c = c * s + s / 2.0
    u = q @ kbar.T + lam * amax[None, :] * erf(sigma * (n[:, None] - p_c[None, :]) / s)
    # a pool cell is selected iff fewer than K pool cells outrank it by (u desc, c asc)
    beats = (u[:, :, None] > u[:, None, :]) | (
        (u[:, :, None] == u[:, None, :]) & (c[None, :, None] < c[None, None, :]))
    urank = np.einsum("nab,na->nb", beats.astype(np.int64), pool.astype(np.int64))
    selected = pool & (urank < K)                                    # [N, C]

    tok_mask = np.repeat(selected, s, axis=1)                        # [N, N]
    o_long, has = masked_softmax_attention(q @ k.T / np.sqrt(d), tok_mask, v)
    rms = np.sqrt((o_long ** 2).mean(axis=1) + rms_eps)
    o_long = np.where(has[:, None], o_long / rms[:, None], 0.0)

    pos = n + pos_offset
    qr, kr = rope_complex(q, pos, rope_base), rope_complex(k, pos, rope_base)
    j = np.arange(N)
    band = (j[None, :] <= n[:, None]) & (j[None, :] > n[:, None] - w)
    o_win, _ = masked_softmax_attention(qr @ kr.T / np.sqrt(d), band, v)

    return dict(out=o_win + mix * o_long, o_win=o_win, o_long=o_long,
                selected=selected, pool=pool, u=u, kbar=kbar, amax=amax)
