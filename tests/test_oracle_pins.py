"""Pins of the fp64 CPU oracle against things other than itself.

Each test checks the oracle against what the FreeSolo pages or mathematics
fix: an independent dense brute force (tests/brute_force.py), textbook
attention from a library routine (torch SDPA in float64), closed forms and
invariants the pages state, and printed constants (tests/golden).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from brute_force import brute_forward, rope_complex
from long_context_lm_gb300.inputs import make_inputs, bf16_values
from oracle import oracle as O

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_constants.json")))
PAGE = dict(w=512, s=32, K=4, P=64, W=8, Bq=128, rope_base=10000.0, rms_eps=1e-6, mode=0)
TINY = dict(w=16, s=4, K=2, P=3, W=2, Bq=8, rope_base=10000.0, rms_eps=1e-6, mode=0)


def head_arrays(inp):
    B, H, N, d = inp.q.shape
    return [bf16_values(t).reshape(B * H, N, d).numpy() for t in (inp.q, inp.k, inp.v)]


def run_oracle(inp, params, rows=None, **kw):
    q, k, v = head_arrays(inp)
    H = inp.q.shape[1]
    return O.forward(q, k, v, H, inp.lam.numpy(), inp.sigma.numpy(), inp.mix.numpy(),
                     rows=rows, params=params, **kw)


def compare_with_brute(inp, params, atol=1e-12):
    q, k, v = head_arrays(inp)
    H = inp.q.shape[1]
    res = run_oracle(inp, params)
    for bh in range(q.shape[0]):
        h = bh % H
        bf = brute_forward(q[bh], k[bh], v[bh], float(inp.lam[h]), float(inp.sigma[h]),
                           float(inp.mix[h]), **params)
        for key in ("out", "o_win", "o_long"):
            np.testing.assert_allclose(res[key][bh], bf[key], atol=atol, rtol=0, err_msg=key)
        sel = res["sel"][bh]
        for n in range(q.shape[1]):
            got = sorted(int(c) for c in sel[n] if c >= 0)
            want = sorted(np.nonzero(bf["selected"][n])[0].tolist())
            assert got == want, (bh, n, got, want)
    return res


# --------------------------------------------------------------------------
# whole forward against the dense brute force
# --------------------------------------------------------------------------

@pytest.mark.parametrize("mode", [0, 1])
def test_brute_force_tiny_params_prunes(mode):
    # s=4, B=8, P=3, W=2, K=2: many blocks with pruning active, so the pool
    # rule, the selection and both softmaxes are all exercised.
    inp = make_inputs(1, 2, 96, head_dim=8, seed=11, sigma_ln=0.8)
    compare_with_brute(inp, dict(TINY, mode=mode))


def test_brute_force_tiny_params_with_norm_ties():
    # Cells whose largest key norm is exactly equal: the pool must break the
    # tie by the older cell first, like the brute force's rank count.
    inp = make_inputs(1, 1, 96, head_dim=8, seed=5)
    k = inp.k.clone()
    base = k[0, 0, 0].clone()
    for t in range(0, 96, 4):       # first token of every cell: same norm
        perm = torch.randperm(8, generator=torch.Generator().manual_seed(t))
        k[0, 0, t] = base[perm] * 3.0
    inp.k = k
    compare_with_brute(inp, TINY)


def test_brute_force_page_params():
    # Page parameters at N=1024: pools equal the whole prefix (see below), K=4.
    inp = make_inputs(1, 2, 1024, seed=3)
    compare_with_brute(inp, PAGE, atol=1e-11)


def test_brute_force_no_erf_term():
    # lambda = 0 (the pages' no-erf ablation): routing by content alone.
    inp = make_inputs(1, 2, 96, head_dim=8, seed=12)
    inp.lam = torch.zeros_like(inp.lam)
    compare_with_brute(inp, TINY)


# --------------------------------------------------------------------------
# window branch: textbook RoPE attention
# --------------------------------------------------------------------------

def test_window_is_textbook_causal_rope_attention():
    # For N <= w every key up to the query is in the window, so with mix = 0
    # the output is plain causal attention on rotated q, k (library SDPA).
    inp = make_inputs(1, 1, 384, seed=7)
    inp.mix = torch.zeros_like(inp.mix)
    q, k, v = head_arrays(inp)
    res = run_oracle(inp, PAGE)
    pos = np.arange(384)
    qr = torch.from_numpy(rope_complex(q[0].astype(np.float64), pos, 10000.0))
    kr = torch.from_numpy(rope_complex(k[0].astype(np.float64), pos, 10000.0))
    ref = torch.nn.functional.scaled_dot_product_attention(
        qr[None], kr[None], torch.from_numpy(v[0].astype(np.float64))[None], is_causal=True)[0]
    np.testing.assert_allclose(res["out"][0], ref.numpy(), atol=1e-12, rtol=0)


def test_window_band_against_sdpa_mask():
    # N > w: a band mask of width w (keys n-w+1 .. n), same library routine.
    p = dict(PAGE, w=64)
    inp = make_inputs(1, 1, 256, seed=8)
    inp.mix = torch.zeros_like(inp.mix)
    q, k, v = head_arrays(inp)
    res = run_oracle(inp, p)
    pos = np.arange(256)
    qr = torch.from_numpy(rope_complex(q[0].astype(np.float64), pos, 10000.0))
    kr = torch.from_numpy(rope_complex(k[0].astype(np.float64), pos, 10000.0))
    i = torch.arange(256)
    band = (i[None, :] <= i[:, None]) & (i[None, :] > i[:, None] - 64)
    ref = torch.nn.functional.scaled_dot_product_attention(
        qr[None], kr[None], torch.from_numpy(v[0].astype(np.float64))[None], attn_mask=band)[0]
    np.testing.assert_allclose(res["out"][0], ref.numpy(), atol=1e-12, rtol=0)


def test_rope_depends_only_on_offset():
    # RoPE makes q_i.k_j a function of j - i (paper.rainbus.top summary,
    # 前置知识): shifting every position by a constant leaves the window
    # branch unchanged.
    inp = make_inputs(1, 1, 640, seed=9)
    a = run_oracle(inp, PAGE, rows=[0, 100, 511, 512, 639])
    b = run_oracle(inp, PAGE, rows=[0, 100, 511, 512, 639], pos_offset=123456.0)
    np.testing.assert_allclose(a["o_win"], b["o_win"], atol=1e-9, rtol=0)
    np.testing.assert_array_equal(a["sel"], b["sel"])


# --------------------------------------------------------------------------
# cell summaries
# --------------------------------------------------------------------------

def test_cell_summaries_against_numpy_and_rotation_invariance():
    inp = make_inputs(1, 2, 512, seed=4)
    _, k, _ = head_arrays(inp)
    kbar, amax = O.cells(k, s=32)
    cells = k.astype(np.float64).reshape(2, 16, 32, 64)
    np.testing.assert_allclose(kbar, cells.mean(axis=2), atol=1e-14, rtol=0)
    np.testing.assert_allclose(amax, np.linalg.norm(cells, axis=3).max(axis=2), rtol=1e-14)
    # a_c is invariant under any rotation of the keys (RoPE is orthogonal)
    rot = rope_complex(k[0].astype(np.float64), np.arange(512) * 7.0 + 3.0, 10000.0)
    _, amax_rot = O.cells(rot[None].astype(np.float32), s=32)
    np.testing.assert_allclose(amax_rot[0], amax[0], rtol=1e-6)
    # a cell of identical keys summarises to that key
    kc = np.tile(k[:1, :1], (1, 64, 1))
    kb1, am1 = O.cells(kc, s=32)
    np.testing.assert_allclose(kb1[0, 0], kc[0, 0], rtol=1e-15)
    np.testing.assert_allclose(am1[0, 0], np.linalg.norm(kc[0, 0].astype(np.float64)), rtol=1e-15)


# --------------------------------------------------------------------------
# pools
# --------------------------------------------------------------------------

@pytest.mark.parametrize("P,W,Bq,s,quant", [(64, 8, 128, 32, 0), (64, 8, 128, 32, 8),
                                            (3, 2, 8, 4, 0), (5, 3, 16, 4, 4), (1, 0, 4, 4, 2)])
def test_running_pool_equals_sorted_definition(P, W, Bq, s, quant):
    # The pruned set of every block equals the top-P by norm over the cells
    # older than the recency window, kept as a running list updated at block
    # boundaries (ai.info summary, Methodology in Plain English).
    rng = np.random.default_rng(P * 100 + W + quant)
    N = Bq * 64
    amax = rng.lognormal(0, 0.5, size=(3, N // s))
    if quant:
        amax = np.round(amax * quant) / quant      # many exact ties
    pd, cd, _ = O.pools(amax, N, s, Bq, P, W, mode=0, streaming=False)
    ps, cs, _ = O.pools(amax, N, s, Bq, P, W, mode=0, streaming=True)
    np.testing.assert_array_equal(cd, cs)
    np.testing.assert_array_equal(pd, ps)
    # size bound: at most P + W cells, every one available
    assert cd.max() <= P + W
    nblk = N // Bq
    for beta in range(nblk):
        A = beta * Bq // s
        ids = pd[:, beta][pd[:, beta] >= 0]
        assert ids.size == 0 or ids.max() < A


def test_pool_size_bound_is_page_value():
    P, W = GOLDEN["prune_P"]["value"], GOLDEN["recent_W"]["value"]
    assert P + W == GOLDEN["pool_max_cells"]["value"]
    rng = np.random.default_rng(0)
    N = 65536
    amax = rng.lognormal(0, 0.5, size=(1, N // 32))
    _, count, _ = O.pools(amax, N)
    assert count.max() == GOLDEN["pool_max_cells"]["value"]


def test_fsl_equals_fs_while_prefix_fits_pool():
    # While the available prefix has at most P+W cells nothing is pruned.
    rng = np.random.default_rng(1)
    N = 8192
    amax = rng.lognormal(0, 0.5, size=(2, N // 32))
    pl, cl, _ = O.pools(amax, N, mode=0)
    pf, cf, _ = O.pools(amax, N, mode=1)
    for beta in range(N // 128):
        A = beta * 4
        same = sorted(pl[0, beta][: cl[0, beta]]) == sorted(pf[0, beta][: cf[0, beta]])
        assert same == (A <= 72), beta


# --------------------------------------------------------------------------
# score: the erf bias and the printed bound
# --------------------------------------------------------------------------

def test_erf_factor_lower_bound_matches_page():
    # With q = 0, lambda = 1, sigma = 4 the score is a_c * g with g the erf
    # factor.  Over every available cell g >= erf(2), and the page prints
    # erf(2) ~ 0.9953 (paper.rainbus.top summary, 局限与改进); the bound is
    # attained by the newest cell for the block's first query.
    gold = GOLDEN["erf_bias_lower_bound"]
    N, d = 1024, 64
    rng = np.random.default_rng(2)
    q1 = np.zeros((N, d), np.float32)
    k1 = rng.standard_normal((N, d)).astype(np.float32)
    _, amax = O.cells(k1[None], s=32)
    gmin = 1.0
    for n in range(128, N, 37):
        pool, u = O.scores(q1, k1, n, lam=1.0, sigma=GOLDEN["sigma_h"]["value"], mode=1)
        g = u / amax[0][pool]
        gmin = min(gmin, g.min())
        assert np.all(g >= math.erf(2.0) - 1e-15)
    b0 = 512
    pool, u = O.scores(q1, k1, b0, lam=1.0, sigma=4.0, mode=1)
    newest = list(pool).index(b0 // 32 - 1)
    g_new = u[newest] / amax[0][pool[newest]]
    assert round(g_new, gold["digits"]) == gold["value"]
    assert round(gmin, gold["digits"]) == gold["value"]


def test_no_erf_term_routes_by_content_alone():
    inp = make_inputs(1, 1, 2048, seed=13)
    inp.lam = torch.zeros_like(inp.lam)
    q, k, _ = head_arrays(inp)
    kbar, _ = O.cells(k, s=32)
    rows = [200, 700, 1500, 2047]
    res = run_oracle(inp, PAGE, rows=rows)
    for r, n in enumerate(rows):
        A = (n // 128) * 4
        dots = kbar[0, :A] @ q[0, n].astype(np.float64)
        want = sorted(np.argsort(-dots, kind="stable")[:4].tolist())
        assert sorted(res["sel"][0, r].tolist()) == want


# --------------------------------------------------------------------------
# readout
# --------------------------------------------------------------------------

def test_block_one_long_branch_is_dense_nope_attention():
    # Block 1 (b0 = 128) has exactly K = 4 available cells, so every query of
    # the block reads tokens 0..127: textbook unrotated attention then RMSNorm.
    inp = make_inputs(1, 1, 512, seed=14)
    q, k, v = head_arrays(inp)
    rows = list(range(128, 256))
    res = run_oracle(inp, PAGE, rows=rows)
    qt = torch.from_numpy(q[0, 128:256].astype(np.float64))[None]
    kt = torch.from_numpy(k[0, :128].astype(np.float64))[None]
    vt = torch.from_numpy(v[0, :128].astype(np.float64))[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)[0].numpy()
    o = o / np.sqrt((o ** 2).mean(axis=1, keepdims=True) + 1e-6)
    np.testing.assert_allclose(res["o_long"][0], o, atol=1e-12, rtol=0)
    # block 0 has no available cell: the long branch is zero
    res0 = run_oracle(inp, PAGE, rows=[0, 5, 127])
    assert np.all(res0["o_long"] == 0) and np.all(res0["sel"] == -1)


def test_read_budget_and_unit_rms():
    inp = make_inputs(1, 2, 4096, seed=15)
    res = run_oracle(inp, PAGE, rows=list(range(0, 4096, 61)))
    nsel = (res["sel"] >= 0).sum(axis=2)
    assert nsel.max() * 32 <= GOLDEN["read_budget_tokens"]["value"]
    # after RMSNorm with eps the RMS is sqrt(ms / (ms + eps)): just below 1
    rms = np.sqrt((res["o_long"] ** 2).mean(axis=2))
    ok = nsel > 0
    assert np.all(rms[ok] <= 1.0 + 1e-12) and np.all(rms[ok] > 0.999)
    assert np.all(rms[~ok] == 0)


def test_mix_is_window_plus_weighted_long_branch():
    inp = make_inputs(1, 2, 1024, seed=16)
    res = run_oracle(inp, PAGE, rows=list(range(0, 1024, 7)))
    mix = inp.mix.numpy()
    np.testing.assert_allclose(res["out"], res["o_win"] + mix[:, None, None] * res["o_long"],
                               atol=1e-13, rtol=0)
    inp.mix = torch.zeros_like(inp.mix)
    res0 = run_oracle(inp, PAGE, rows=list(range(0, 1024, 7)))
    np.testing.assert_allclose(res0["out"], res0["o_win"], atol=0, rtol=0)


# --------------------------------------------------------------------------
# causality and retrieval
# --------------------------------------------------------------------------

def test_future_tokens_do_not_change_a_row():
    inp = make_inputs(1, 1, 2048, seed=17)
    rows = [130, 777, 1500]
    a = run_oracle(inp, PAGE, rows=rows)
    for n in rows:
        pert = make_inputs(1, 1, 2048, seed=18)
        inp2 = make_inputs(1, 1, 2048, seed=17)
        for name in ("q", "k", "v"):
            t = getattr(inp2, name).clone()
            t[:, :, n + 1:] = getattr(pert, name)[:, :, n + 1:]
            setattr(inp2, name, t)
        b = run_oracle(inp2, PAGE, rows=[n])
        r = rows.index(n)
        np.testing.assert_array_equal(a["out"][:, r], b["out"][:, 0])
        np.testing.assert_array_equal(a["sel"][:, r], b["sel"][:, 0])


def test_selected_cells_end_before_block_start():
    inp = make_inputs(1, 2, 8192, seed=19)
    rows = list(range(0, 8192, 29))
    res = run_oracle(inp, PAGE, rows=rows)
    for r, n in enumerate(rows):
        b0 = (n // 128) * 128
        ids = res["sel"][:, r][res["sel"][:, r] >= 0]
        assert np.all((ids + 1) * 32 <= b0)


@pytest.mark.parametrize("seed", [20, 21, 22])
def test_planted_needle_is_selected(seed):
    # A key planted as 12x a later query (3x the query with its norm boosted
    # 4x, the single-needle probe of the pages, 实验结果) survives pruning and
    # must be among that query's K cells.
    inp = make_inputs(1, 4, 8192, seed=seed, needles="deep", n_needles=1)
    rows = sorted({j for (_, _, _, j) in inp.needles})
    res = run_oracle(inp, PAGE, rows=rows)
    H = 4
    for (b, h, p, j) in inp.needles:
        bh = b * H + h
        assert p // 32 in res["sel"][bh, rows.index(j)].tolist(), (h, p, j)
