"""Pins of the FS-B selection oracle (oracle/fsb.py) against things other than
itself: the node bound holds for every cell beneath every node; a beam wide
enough to keep every node reduces the search to brute force over the
available cells (ranked with scipy's logsumexp, a library routine); small
prefixes never lose a cell; causality; a planted needle is found by the
page beam of 16; the two forests coincide when tau admits every cell."""
import math

import numpy as np
import pytest
from scipy.special import logsumexp

from oracle import fsb


def _head(C, d=16, s=4, seed=0, spread=0.8):
    rng = np.random.default_rng(seed)
    N = C * s
    k = rng.standard_normal((N, d)) * np.exp(spread * rng.standard_normal((N, 1)))
    kbar = k.reshape(C, s, d).mean(1)
    amax = np.linalg.norm(k, axis=1).reshape(C, s).max(1)
    q = rng.standard_normal((N, d))
    return q, k, kbar, amax


def _cell_score(q, kbar, amax, c, n, lam, sigma, s):
    return float(q @ kbar[c]) + lam * amax[c] * math.erf(sigma * (n - (c * s + s / 2)) / s)


def test_node_bound_covers_every_cell_beneath():
    s, C = 4, 45
    q, k, kbar, amax = _head(C, s=s, seed=1)
    cells = np.arange(C)
    levels = fsb.build_forest(cells, kbar, amax)
    for n in (C * s - 1, C * s + 37):
        for lam in (0.5, 1.5):
            for j, lev in enumerate(levels):
                for i in range(len(lev["mean"])):
                    lo, hi = i << j, min(C, (i + 1) << j)
                    ub = fsb.node_bound(q[n % (C * s)], lev, i, n, lam, 4.0, s)
                    best = max(_cell_score(q[n % (C * s)], kbar, amax, c, n, lam, 4.0, s)
                               for c in cells[lo:hi])
                    assert ub >= best - 1e-12, (j, i, ub, best)
    # a leaf's bound is the cell's score itself
    assert abs(fsb.node_bound(q[7], levels[0], 3, 200, 1.0, 4.0, s)
               - _cell_score(q[7], kbar, amax, 3, 200, 1.0, 4.0, s)) < 1e-12


def _brute(q, k, n, A, K, s):
    lse = [(-float(logsumexp(k[c * s:(c + 1) * s] @ q / math.sqrt(q.shape[0]))), c)
           for c in range(A)]
    return [c for _, c in sorted(lse)[:K]]


@pytest.mark.parametrize("tau", [-1.0, 3.0, np.inf])
def test_unbounded_beam_is_brute_force(tau):
    s, Bq, K, C = 4, 8, 3, 64
    q, k, kbar, amax = _head(C, s=s, seed=2)
    for n in (9, 40, 133, 255):
        sel, _, _ = fsb.fsb_select_row(q[n], k, kbar, amax, n, 1.0, 4.0, tau, s=s, Bq=Bq, K=K,
                                       beam=10 ** 6)
        A = (n // Bq) * Bq // s
        assert sel == _brute(q[n], k, n, A, K, s), (n, sel)


def test_small_prefix_keeps_every_cell_with_the_page_beam():
    # at most 16 available cells: no level of either forest has more than 16
    # nodes, so the page beam drops nothing
    s, Bq, K, C = 4, 8, 4, 40
    q, k, kbar, amax = _head(C, s=s, seed=3)
    for n in range(8, 8 * 9, 5):  # A <= 16
        sel, gap, _ = fsb.fsb_select_row(q[n], k, kbar, amax, n, 1.0, 4.0, 2.0, s=s, Bq=Bq,
                                         K=K, beam=16)
        A = (n // Bq) * Bq // s
        assert sel == _brute(q[n], k, n, A, K, s)
        assert gap == math.inf


def test_causality_and_block_zero():
    s, Bq, C = 32, 128, 40
    q, k, kbar, amax = _head(C, d=64, s=s, seed=4)
    for n in (0, 127, 128, 700, 1279):
        sel, _, _ = fsb.fsb_select_row(q[n], k, kbar, amax, n, 1.0, 4.0, 8.0)
        A = (n // Bq) * Bq // s
        assert all(0 <= c < A for c in sel)
        assert len(sel) == min(4, A)


def test_both_forests_coincide_when_tau_admits_every_cell():
    s, C = 32, 96
    q, k, kbar, amax = _head(C, d=64, s=s, seed=5)
    n = C * s - 1
    A = (n // 128) * 128 // s
    lv = fsb.build_forest(np.arange(A), kbar, amax)
    full, _ = fsb.beam_search(q[n], lv, A, n, 1.0, 4.0, s, 16)
    sel_all, _, _ = fsb.fsb_select_row(q[n], k, kbar, amax, n, 1.0, 4.0, -1.0)
    sel_full, _, _ = fsb.fsb_select_row(q[n], k, kbar, amax, n, 1.0, 4.0, np.inf)
    assert sel_all == sel_full
    assert set(sel_full) <= set(full)


def test_needle_found_with_the_page_beam():
    s, C, d = 32, 512, 64
    rng = np.random.default_rng(6)
    q, k, kbar, amax = _head(C, d=d, s=s, seed=6, spread=0.5)
    n = C * s - 1
    for trial in range(5):
        c0 = int(rng.integers(0, C // 2))
        kk = k.copy()
        kk[c0 * s + 7] = 12.0 * q[n]  # a key far along the query, with a large norm
        kb = kk.reshape(C, s, d).mean(1)
        am = np.linalg.norm(kk, axis=1).reshape(C, s).max(1)
        tau = float(np.median(am))
        sel, _, _ = fsb.fsb_select_row(q[n], kk, kb, am, n, 1.0, 4.0, tau)
        assert c0 in sel, (trial, c0, sel)
