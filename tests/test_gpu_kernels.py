"""Per-kernel parity of the CUDA path against the fp64 oracle (GPU only).

Each kernel is called through the C ABI (long_context_lm_gb300.fs) on seeded
synthetic inputs spanning several tiles and compared element by element with
the oracle stage it implements."""
import numpy as np
import pytest
import torch

from long_context_lm_gb300 import fs
from long_context_lm_gb300.inputs import make_inputs
from oracle import oracle as O
from parity import (MAX_ABS, MEAN_ABS, compare_forward, head_slices, oracle_rows, sample_rows,
                    to_device)

pytestmark = pytest.mark.gpu
PAGE = dict(w=512, s=32, K=4, P=64, W=8, Bq=128, rope_base=10000.0, rms_eps=1e-6, mode=0)


# --------------------------------------------------------------------------- K1
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("B,H,N", [(1, 1, 128), (2, 3, 4096), (1, 2, 8192 + 128)])
def test_cell_summary(dtype, B, H, N):
    inp = make_inputs(B, H, N, seed=N + H, sigma_ln=0.8, dtype=dtype)
    kbar, amax = fs.fs_cell_summarize(inp.k.cuda())
    _, k, _ = head_slices(inp)
    rk, ra = O.cells(k, s=32)
    kb = kbar.cpu().numpy().reshape(rk.shape)
    am = amax.cpu().numpy().reshape(ra.shape)
    np.testing.assert_allclose(kb, rk, rtol=0, atol=2e-6 * np.abs(rk).max())
    np.testing.assert_allclose(am, ra, rtol=2e-6, atol=0)


# --------------------------------------------------------------------------- K2
def _gpu_pools(amax_np, N, P, W):
    amax = torch.from_numpy(amax_np.astype(np.float32)).cuda()[None]
    pool, count = fs.fs_prune_cells(amax, N, dict(P=P, W=W))
    return pool[0].cpu().numpy(), count[0].cpu().numpy()


# 393216: 192 chunks of 64 cells, the most the per-head shared-memory scan takes;
# 401408: past it, the two global-memory kernels
@pytest.mark.parametrize("N", [128, 256, 2304, 2432, 8192, 65536, 262144 + 128, 393216, 401408])
@pytest.mark.parametrize("P,W,quant", [(64, 8, 0), (64, 8, 4), (3, 2, 0), (64, 0, 2), (1, 8, 0)])
def test_prune_is_bit_exact(N, P, W, quant):
    # Integer/index work: identical to the oracle's definition (sort per
    # block) on the same norms, in the same order, including exact ties.
    rng = np.random.default_rng(N + P + W + quant)
    H = 3
    amax = rng.lognormal(0, 0.5, size=(H, N // 32)).astype(np.float32)
    if quant:
        amax = (np.round(amax * quant) / quant).astype(np.float32)
    pool, count = _gpu_pools(amax, N, P, W)
    ref_pool, ref_count, _ = O.pools(amax.astype(np.float64), N, 32, 128, P, W, mode=0)
    np.testing.assert_array_equal(count, ref_count)
    np.testing.assert_array_equal(pool, ref_pool)


# --------------------------------------------------------------------------- K3
def _select(inp, params, with_scores=False):
    d = to_device(inp)
    kbar, amax = fs.fs_cell_summarize(d["k"])
    pool = count = None
    if params.get("mode", 0) == 0:
        pool, count = fs.fs_prune_cells(amax, inp.q.shape[2], params)
    return fs.fs_select_cells(d["q"], kbar, amax, pool, count, d["lam"], d["sigma"], params,
                              with_scores=with_scores)


@pytest.mark.parametrize("params,N,lam0", [
    (PAGE, 8192, False),
    (dict(PAGE, mode=1), 4096, False),
    (dict(PAGE, mode=1), 16384, False),   # up to 508 candidates: four 128-cell chunks
    (PAGE, 4096, True),
    (dict(PAGE, K=1), 4096, False),
    (dict(PAGE, K=8, P=16, W=2), 8192, False),
])
def test_select_matches_oracle(params, N, lam0):
    inp = make_inputs(1, 4, N, seed=N + params["K"], sigma_ln=0.8)
    if lam0:
        inp.lam = torch.zeros_like(inp.lam)
    sel, score = _select(inp, params, with_scores=True)
    sel = sel.cpu().numpy().reshape(4, N, -1)
    score = score.cpu().numpy().reshape(4, N, -1)
    rows = sample_rows(N, n_blocks=24, per_block=24, seed=1)
    ref = oracle_rows(inp, rows, params)
    ties = 0
    for bh in range(4):
        for i, n in enumerate(rows):
            a = [int(c) for c in sel[bh, n]]
            b = [int(c) for c in ref["sel"][bh, i]]
            if sorted(a) != sorted(b):
                assert min(ref["gap_rel"][bh, i], ref["pool_gap"][bh, i]) < 1e-5, (bh, n, a, b)
                ties += 1
                continue
            if a != b:  # same set, different rank order: only on near-equal scores
                np.testing.assert_allclose(np.sort(score[bh, n]), np.sort(ref["sel_score"][bh, i]),
                                           rtol=1e-5)
            valid = np.asarray(b) >= 0
            np.testing.assert_allclose(np.sort(score[bh, n][valid]),
                                       np.sort(ref["sel_score"][bh, i][valid]), rtol=2e-6, atol=2e-5)
    assert ties <= 1e-3 * 4 * len(rows)


# --------------------------------------------------------------------------- K4
@pytest.mark.parametrize("N,K", [(4096, 4), (8192, 8), (1024, 1)])
def test_readout_on_given_selection(N, K):
    # The kernel's own selection is fed to both sides, so this checks the
    # gathered NoPE softmax + RMSNorm alone.
    params = dict(PAGE, K=K)
    inp = make_inputs(1, 2, N, seed=40 + K, sigma_ln=0.8, needles="uniform" if N > 2048 else "none",
                      n_needles=4)
    d = to_device(inp)
    sel = _select(inp, params)
    o_long = fs.fs_sparse_readout(d["q"], d["k"], d["v"], sel, params)
    sel_np = sel.cpu().numpy().reshape(2, N, K)
    ol = o_long.cpu().numpy().reshape(2, N, 64)
    q, k, v = head_slices(inp)
    rows = sample_rows(N, n_blocks=20, per_block=16, seed=2)
    err = []
    for bh in range(2):
        for n in rows:
            ref = O.readout(q[bh], k[bh], v[bh], int(n), sel_np[bh, n].tolist())
            err.append(np.abs(ol[bh, n] - ref))
    err = np.array(err)
    assert err.max() < 2e-4 and err.mean() < 2e-5, (err.max(), err.mean())


def test_readout_adversarial_union():
    # Every query of a block picks different cells (large union): forced by
    # a hand-built selection so the union holds many cells.
    N, K = 4096, 4
    inp = make_inputs(1, 1, N, seed=77)
    d = to_device(inp)
    rng = np.random.default_rng(3)
    sel = np.full((1, 1, N, K), -1, np.int32)
    for n in range(N):
        A = (n // 128) * 4
        if A:
            sel[0, 0, n, :min(K, A)] = rng.choice(A, size=min(K, A), replace=False)
    o_long = fs.fs_sparse_readout(d["q"], d["k"], d["v"], torch.from_numpy(sel).cuda(), PAGE)
    ol = o_long.cpu().numpy()[0, 0]
    q, k, v = head_slices(inp)
    for n in sample_rows(N, 12, 12, seed=4):
        ref = O.readout(q[0], k[0], v[0], int(n), sel[0, 0, n].tolist())
        np.testing.assert_allclose(ol[n], ref, atol=2e-4, rtol=0)


@pytest.mark.parametrize("K", [4, 8])
def test_readout_union_wider_than_8192_cells(K):
    # Past N = 8192 * s a block's selections can span more than 8192 cell ids,
    # and the kernel's union is then built window by window.  Each row picks
    # K cells spread over the whole history; half the rows of a block share
    # their first cell (duplicates across rows, across the window edges too).
    N = 262144 + 16384
    inp = make_inputs(1, 1, N, seed=91 + K)
    d = to_device(inp)
    rng = np.random.default_rng(K)
    n = np.arange(N)
    A = (n // 128) * 4
    c0 = np.floor(rng.random(N) * np.maximum(A, 1)).astype(np.int64)
    shared = np.floor(rng.random(N // 128) * np.maximum(A[::128], 1)).astype(np.int64)
    c0 = np.where(n % 2 == 0, shared[n // 128], c0)
    step = np.maximum(A // K, 1)
    sel = np.stack([(c0 + j * step) % np.maximum(A, 1) for j in range(K)], axis=1)
    sel = np.where(A[:, None] >= K, sel, -1).astype(np.int32)
    o_long = fs.fs_sparse_readout(d["q"], d["k"], d["v"],
                                  torch.from_numpy(sel).view(1, 1, N, K).cuda(), dict(PAGE, K=K))
    ol = o_long.cpu().numpy()[0, 0]
    q, k, v = head_slices(inp)
    rows = np.unique(np.concatenate([sample_rows(N, 10, 8, seed=K),
                                     N - 128 + np.arange(0, 128, 9), [N - 1]]))
    for r in rows:
        ref = O.readout(q[0], k[0], v[0], int(r), sel[r].tolist())
        np.testing.assert_allclose(ol[r], ref, atol=2e-4, rtol=0)


# --------------------------------------------------------------------------- K5
@pytest.mark.parametrize("N,w", [(128, 512), (1024, 512), (4096, 512), (2048, 1), (2048, 64),
                                 (2048, 100), (4096, 1000)])
def test_window_matches_oracle(N, w):
    params = dict(PAGE, w=w)
    inp = make_inputs(2, 2, N, seed=N + w, sigma_ln=0.8)
    d = to_device(inp)
    out = fs.fs_window_attn(d["q"], d["k"], d["v"], None, None, params)
    rows = sample_rows(N, n_blocks=16, per_block=16, seed=5)
    ref = oracle_rows(inp, rows, params)
    got = out.cpu().numpy().reshape(4, N, 64)[:, rows]
    err = np.abs(got - ref["o_win"])
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (err.max(), err.mean())
    if w == 1:  # window of the token itself: o_win = v_n exactly
        _, _, v = head_slices(inp)
        np.testing.assert_allclose(got, v[:, rows], atol=1e-6, rtol=0)


def test_window_mix_epilogue():
    N = 2048
    inp = make_inputs(1, 2, N, seed=9)
    d = to_device(inp)
    o_long = torch.randn(1, 2, N, 64, device="cuda")
    a = fs.fs_window_attn(d["q"], d["k"], d["v"], None, None, PAGE)
    b = fs.fs_window_attn(d["q"], d["k"], d["v"], o_long, d["mix"], PAGE)
    torch.testing.assert_close(b, a + d["mix"][None, :, None, None] * o_long, atol=1e-6, rtol=1e-6)
