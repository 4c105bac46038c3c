"""Gradients of the FS-L forward on the GPU (fs_attention_bwd) against the
fp64 oracle's backward (pinned by finite differences and float64 autograd in
test_oracle_backward.py), GPU only.

Both sides hold the pools and selections at the forward's; the test first
checks that the GPU forward selects the oracle's cells on every row (so
both differentiate the same function).  Tolerance from the arithmetic: the
GPU takes every product on the tensor cores with fp32 accumulation, its
fp32 operands (rotated q and k, g, P, dS, do) split into bf16 hi + lo and
multiplied as hi.hi + hi.lo + lo.hi (about 2^-16 relative per product; bf16
q, k, v are exact), over up to w + K*s products per row and about w + 128
per key, with fast exponentials (relative error about 2^-21).  The test
allows max-abs 2e-4 and mean-abs 2e-5 relative to each gradient's largest
magnitude."""
import numpy as np
import pytest
import torch

from long_context_lm_gb300 import fs
from long_context_lm_gb300.inputs import bf16_values, make_inputs
from oracle import oracle as O
from parity import to_device

pytestmark = pytest.mark.gpu
PAGE = dict(w=512, s=32, K=4, P=64, W=8, Bq=128, rope_base=10000.0, rms_eps=1e-6, mode=0)


def _run(B, H, N, params, seed, sigma_ln=0.8):
    inp = make_inputs(B, H, N, seed=seed, sigma_ln=sigma_ln)
    d = to_device(inp)
    gen = torch.Generator().manual_seed(seed + 1)
    g = torch.randn((B, H, N, 64), generator=gen, dtype=torch.float32)
    # the forward's selection equals the oracle's on every row
    ws = torch.empty(fs.fs_workspace_bytes(B, H, N, 64, params), device="cuda", dtype=torch.uint8)
    fs.fs_attention_fwd(d["q"], d["k"], d["v"], d["lam"], d["sigma"], d["mix"], params, ws=ws)
    sel = fs.fs_workspace_view(ws, B, H, N, 64, params)["sel"].cpu().numpy().reshape(B * H, N, -1)
    q, k, v = [bf16_values(t).reshape(B * H, N, 64).numpy() for t in (inp.q, inp.k, inp.v)]
    ref_f = O.forward(q, k, v, H, inp.lam.numpy(), inp.sigma.numpy(), inp.mix.numpy(),
                      params=params, want_branches=False)
    for bh in range(B * H):
        for n in range(N):
            assert sorted(sel[bh, n].tolist()) == sorted(ref_f["sel"][bh, n].tolist()), (bh, n)
    dq, dk, dv, dmix = fs.fs_attention_bwd(d["q"], d["k"], d["v"], d["lam"], d["sigma"], d["mix"],
                                           g.cuda(), params)
    fs.fs_check_status(ws)
    torch.cuda.synchronize()
    ref = O.backward(q, k, v, H, inp.lam.numpy(), inp.sigma.numpy(), inp.mix.numpy(),
                     g.numpy().reshape(B * H, N, 64), params=params)
    got = dict(dq=dq, dk=dk, dv=dv)
    stats = {}
    for name in ("dq", "dk", "dv"):
        a = got[name].cpu().numpy().reshape(B * H, N, 64).astype(np.float64)
        r = ref[name]
        scale = np.abs(r).max()
        err = np.abs(a - r)
        stats[name] = (float(err.max() / scale), float(err.mean() / scale))
        assert err.max() <= 2e-4 * scale and err.mean() <= 2e-5 * scale, (name, stats[name])
    np.testing.assert_allclose(dmix.cpu().numpy(), ref["dmix"], rtol=1e-4,
                               atol=1e-4 * np.abs(ref["dmix"]).max())
    return stats


@pytest.mark.parametrize("B,H,N,params,seed", [
    (1, 2, 1024, PAGE, 0),
    (2, 2, 768, dict(PAGE, w=64, K=2, P=8, W=2), 1),   # pruning active, small window
    (1, 2, 640, dict(PAGE, mode=1), 2),                # base FS (every available cell)
    (1, 1, 2560, PAGE, 3),                             # the pool is pruned (A > 72)
    (1, 2, 256, dict(PAGE, K=8), 4),                   # K = 8
    # unions of several long tiles; a seed whose selections have no near tie
    # (smallest deciding gap 6.8e-5 relative), so both sides pick the same cells
    (1, 2, 4096, PAGE, 19),
    (1, 1, 1024, dict(PAGE, w=200), 6),                # window edge inside a tile
    (1, 1, 512, dict(PAGE, w=1), 7),                   # the window is the token itself
    (1, 2, 1024, dict(PAGE, K=1), 8),                  # one cell per row
])
def test_backward_matches_oracle(B, H, N, params, seed):
    print(_run(B, H, N, params, seed))
