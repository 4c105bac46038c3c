"""Shared comparison logic of the GPU parity tests (CUDA path vs fp64 oracle).

Rules (fixed by the accuracy contract of this implementation):
  * cell indices (pools, selections) must match exactly, except where the
    oracle's deciding gap -- K-th vs (K+1)-th score, or the P-th vs (P+1)-th
    older-cell norm that fixed the pool -- is below 1e-5 relative; such rows
    are counted and must stay under 0.1% of the compared rows, and their
    output is checked against the oracle's readout of the kernel's own
    selection;
  * outputs must be within max-abs 1e-2 and mean-abs 1e-3 of the oracle.
"""
from __future__ import annotations

import numpy as np
import torch

from long_context_lm_gb300.inputs import bf16_values
from oracle import oracle as O

TIE_REL = 1e-5
TIE_FRACTION = 1e-3
MAX_ABS = 1e-2
MEAN_ABS = 1e-3


def head_slices(inp):
    """bf16-rounded q, k, v as float32 numpy [BH, N, d]."""
    B, H, N, d = inp.q.shape
    return [bf16_values(t).reshape(B * H, N, d).numpy() for t in (inp.q, inp.k, inp.v)]


def to_device(inp, dev="cuda"):
    return dict(q=inp.q.to(dev), k=inp.k.to(dev), v=inp.v.to(dev), lam=inp.lam.to(dev),
                sigma=inp.sigma.to(dev), mix=inp.mix.to(dev))


def oracle_rows(inp, rows, params, nthreads=0):
    """Oracle forward for the given rows of every head, one head at a time
    (bounds host memory at long N).  rows: 1-D array used for every head."""
    q, k, v = head_slices(inp)
    H = inp.q.shape[1]
    BH = q.shape[0]
    outs = []
    for bh in range(BH):
        h = bh % H
        r = O.forward(q[bh:bh + 1], k[bh:bh + 1], v[bh:bh + 1], 1, inp.lam.numpy()[h:h + 1],
                      inp.sigma.numpy()[h:h + 1], inp.mix.numpy()[h:h + 1], rows=rows,
                      params=params, nthreads=nthreads)
        outs.append(r)
    return {key: np.concatenate([o[key] for o in outs], axis=0) for key in outs[0]}


def compare_forward(inp, params, rows, gpu_out, gpu_sel, ref=None, check_sel=True):
    """gpu_out [BH, N, d], gpu_sel [BH, N, K] (numpy) vs the oracle on `rows`.
    Returns a stats dict; raises AssertionError on a violation."""
    rows = np.asarray(rows)
    if ref is None:
        ref = oracle_rows(inp, rows, params)
    q, k, v = head_slices(inp)
    H = inp.q.shape[1]
    BH = gpu_out.shape[0]
    s = params.get("s", 32)
    eps = params.get("rms_eps", 1e-6)
    out_g = gpu_out[:, rows]
    ref_out = ref["out"].copy()
    n_tie = n_hard = 0
    hard = []
    if check_sel:
        sel_g = gpu_sel[:, rows]
        for bh in range(BH):
            for i, n in enumerate(rows):
                a = sorted(int(c) for c in sel_g[bh, i] if c >= 0)
                b = sorted(int(c) for c in ref["sel"][bh, i] if c >= 0)
                if a == b:
                    continue
                gap = min(ref["gap_rel"][bh, i], ref["pool_gap"][bh, i])
                if gap < TIE_REL:
                    n_tie += 1
                    h = bh % H
                    ol = O.readout(q[bh], k[bh], v[bh], int(n), a, s=s, eps=eps)
                    ref_out[bh, i] = ref["o_win"][bh, i] + float(inp.mix[h]) * ol
                else:
                    n_hard += 1
                    if len(hard) < 5:
                        hard.append((bh, int(n), a, b, float(gap)))
    total = BH * len(rows)
    err = np.abs(out_g.astype(np.float64) - ref_out)
    stats = dict(rows=total, tie_mismatch=n_tie, hard_mismatch=n_hard,
                 max_abs=float(err.max()), mean_abs=float(err.mean()))
    assert n_hard == 0, f"selection mismatches without a near tie: {hard}"
    assert n_tie <= TIE_FRACTION * total, stats
    assert stats["max_abs"] <= MAX_ABS, stats
    assert stats["mean_abs"] <= MEAN_ABS, stats
    return stats


def sample_rows(N, n_blocks=24, per_block=16, seed=0, Bq=128):
    """Rows spread over blocks (first, last and random ones), with the first
    and last row of each chosen block and random rows inside it."""
    rng = np.random.default_rng(seed)
    nblk = N // Bq
    blocks = sorted(b for b in set([0, 1, 2, nblk - 1] +
                                   rng.integers(0, nblk, size=max(0, n_blocks - 4)).tolist())
                    if 0 <= b < nblk)
    rows = []
    for b in blocks:
        rows += [b * Bq, b * Bq + Bq - 1]
        rows += (b * Bq + rng.integers(0, Bq, size=per_block - 2)).tolist()
    return np.unique(np.asarray(rows, dtype=np.int64))
