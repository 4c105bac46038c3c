"""ctypes front end of the fp64 CPU oracle in ``fs_oracle.c`` (forward, and the
backward with the hard indices held fixed).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg call this module.  The product path
(``long_context_lm_gb300``) never imports it, and this module imports nothing
from the product.

The oracle follows the FreeSolo paper summaries ("FreeSolo: Linear-time Sparse
Attention with Zero-Shot Length Extrapolation": paper.rainbus.top summary,
核心方法 / 方法步骤详情 ②-⑥; ai.info summary, "Methodology in Plain English").
Every function below takes arrays shaped ``[BH, N, d]`` (one slice per
(batch, head) pair) holding bf16-rounded values as float32.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "fs_oracle.c")
LIB = os.path.join(HERE, "libfs_oracle.so")

DEFAULT_PARAMS = dict(w=512, s=32, K=4, P=64, W=8, Bq=128, rope_base=10000.0,
                      rms_eps=1e-6, mode=0)

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, no fast-math) next to its source."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp, SRC, "-lm"])
        os.replace(tmp, LIB)
    return LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i, dbl = ctypes.c_int, ctypes.c_double
            L.fso_cells.argtypes = [P, i, i, i, i, P, P, i]
            L.fso_pools.argtypes = [P, i, i, i, i, i, i, i, i, P, P, P, i, i]
            L.fso_scores.argtypes = [P, P, i, i, i, i, i, i, i, dbl, dbl, i, P, P]
            L.fso_readout.argtypes = [P, P, P, i, i, i, i, P, i, dbl, P]
            L.fso_forward.argtypes = ([P, P, P, i, i, i, i, i, i, i, i, i, i,
                                       dbl, dbl, i, dbl, P, P, P, P, i]
                                      + [P] * 7 + [i])
            L.fso_backward.argtypes = ([P, P, P, i, i, i, i, i, i, i, i, i, i,
                                        dbl, dbl, i, P, P, P, P, P, P, P, P, i])
            L.fso_max_threads.restype = i
            _lib = L
    return _lib


def _f32(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return lib().fso_max_threads()


def cells(k, s=32, nthreads=0):
    """kbar [BH, N/s, d] and amax [BH, N/s] of keys k [BH, N, d]."""
    k = _f32(k)
    BH, N, d = k.shape
    C = N // s
    kbar = np.zeros((BH, C, d), np.float64)
    amax = np.zeros((BH, C), np.float64)
    rc = lib().fso_cells(_ptr(k), BH, N, d, s, _ptr(kbar), _ptr(amax), nthreads)
    assert rc == 0, rc
    return kbar, amax


def pools(amax, N, s=32, Bq=128, P=64, W=8, mode=0, streaming=False, nthreads=0):
    """Pools of every query block.  Returns (pool [BH, nblk, cap] int32 padded
    with -1, count [BH, nblk], gap_rel [BH, nblk]).  Pool order: recent cells
    ascending, then the kept older cells by (a desc, c asc)."""
    amax = np.ascontiguousarray(amax, dtype=np.float64)
    BH = amax.shape[0]
    nblk = N // Bq
    cap = max(1, (nblk - 1) * Bq // s) if mode == 1 else P + W
    pool = np.full((BH, nblk, cap), -1, np.int32)
    count = np.zeros((BH, nblk), np.int32)
    gap = np.full((BH, nblk), np.inf)
    rc = lib().fso_pools(_ptr(amax), BH, N, s, Bq, P, W, mode, int(streaming),
                         _ptr(pool), _ptr(count), None if streaming else _ptr(gap),
                         cap, nthreads)
    assert rc == 0, rc
    return pool, count, gap


def scores(q1, k1, n, lam, sigma, s=32, Bq=128, P=64, W=8, mode=0):
    """Pool of query n's block and the score u of each pool cell (one head)."""
    q1, k1 = _f32(q1), _f32(k1)
    N, d = q1.shape
    C = N // s
    pool = np.full(C + 1, -1, np.int32)
    u = np.zeros(C + 1, np.float64)
    npool = lib().fso_scores(_ptr(q1), _ptr(k1), N, d, s, Bq, P, W, mode,
                             float(lam), float(sigma), int(n), _ptr(pool), _ptr(u))
    return pool[:npool].copy(), u[:npool].copy()


def readout(q1, k1, v1, n, sel, s=32, eps=1e-6):
    """NoPE readout + RMSNorm of query n over the cells in ``sel`` (one head)."""
    q1, k1, v1 = _f32(q1), _f32(k1), _f32(v1)
    N, d = q1.shape
    sel = np.ascontiguousarray([c for c in sel if c >= 0], dtype=np.int32)
    o = np.zeros(d, np.float64)
    lib().fso_readout(_ptr(q1), _ptr(k1), _ptr(v1), N, d, s, int(n), _ptr(sel),
                      len(sel), float(eps), _ptr(o))
    return o


def forward(q, k, v, H, lam, sigma, mix, rows=None, params=None, pos_offset=0.0,
            nthreads=0, want_branches=True):
    """Oracle forward for the requested rows of every [BH, N, d] head slice.

    Returns a dict with ``out``, ``o_win``, ``o_long`` [BH, R, d] (float64),
    ``sel`` [BH, R, K] (int32, -1 padded, ranked), ``sel_score`` [BH, R, K],
    ``gap_rel`` [BH, R] (relative gap of the K-th vs (K+1)-th score) and
    ``pool_gap`` [BH, R] (relative norm gap that fixed the row's pool)."""
    p = dict(DEFAULT_PARAMS)
    if params:
        p.update(params)
    q, k, v = _f32(q), _f32(k), _f32(v)
    BH, N, d = q.shape
    lam = np.ascontiguousarray(lam, dtype=np.float64).reshape(-1)
    sigma = np.ascontiguousarray(sigma, dtype=np.float64).reshape(-1)
    mix = np.ascontiguousarray(mix, dtype=np.float64).reshape(-1)
    assert lam.size == H and sigma.size == H and mix.size == H and BH % H == 0
    if rows is None:
        R, rows_arr = N, None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1)
        R = rows_arr.size
    K = p["K"]
    res = dict(out=np.zeros((BH, R, d)), sel=np.zeros((BH, R, K), np.int32),
               sel_score=np.zeros((BH, R, K)), gap_rel=np.zeros((BH, R)),
               pool_gap=np.zeros((BH, R)))
    if want_branches:
        res["o_win"] = np.zeros((BH, R, d))
        res["o_long"] = np.zeros((BH, R, d))
    rc = lib().fso_forward(
        _ptr(q), _ptr(k), _ptr(v), BH, H, N, d, p["w"], p["s"], K, p["P"], p["W"],
        p["Bq"], float(p["rope_base"]), float(p["rms_eps"]), int(p["mode"]),
        float(pos_offset), _ptr(lam), _ptr(sigma), _ptr(mix), _ptr(rows_arr), R,
        _ptr(res["out"]), _ptr(res.get("o_win")), _ptr(res.get("o_long")),
        _ptr(res["sel"]), _ptr(res["sel_score"]), _ptr(res["gap_rel"]),
        _ptr(res["pool_gap"]), nthreads)
    assert rc == 0, rc
    return res


def backward(q, k, v, H, lam, sigma, mix, g, params=None, nthreads=0):
    """Gradients of L = sum(g * out) for the forward of every [BH, N, d] head
    slice, with the pools and selections held fixed (the pages: hard top-P /
    top-K indices carry no gradient; sigma_h, lambda_h fixed).  Returns a dict
    with ``dq``, ``dk``, ``dv`` [BH, N, d] and ``dmix`` [H] (float64)."""
    p = dict(DEFAULT_PARAMS)
    if params:
        p.update(params)
    q, k, v = _f32(q), _f32(k), _f32(v)
    BH, N, d = q.shape
    g = np.ascontiguousarray(g, dtype=np.float64)
    assert g.shape == q.shape
    lam = np.ascontiguousarray(lam, dtype=np.float64).reshape(-1)
    sigma = np.ascontiguousarray(sigma, dtype=np.float64).reshape(-1)
    mix = np.ascontiguousarray(mix, dtype=np.float64).reshape(-1)
    assert lam.size == H and sigma.size == H and mix.size == H and BH % H == 0
    res = dict(dq=np.zeros((BH, N, d)), dk=np.zeros((BH, N, d)), dv=np.zeros((BH, N, d)),
               dmix=np.zeros(H))
    rc = lib().fso_backward(
        _ptr(q), _ptr(k), _ptr(v), BH, H, N, d, p["w"], p["s"], p["K"], p["P"], p["W"],
        p["Bq"], float(p["rope_base"]), float(p["rms_eps"]), int(p["mode"]),
        _ptr(lam), _ptr(sigma), _ptr(mix), _ptr(g), _ptr(res["dq"]), _ptr(res["dk"]),
        _ptr(res["dv"]), _ptr(res["dmix"]), nthreads)
    assert rc == 0, rc
    return res
