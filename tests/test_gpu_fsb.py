"""FS-B selection and the FS-B forward on the GPU against the fp64 oracle
(oracle/fsb.py for the selection; the oracle's readout, window branch and mix
for the rest), GPU only.

Selections must match exactly except where a decision was a near tie in the
oracle: the gap between the last kept and the first dropped node bound at
some level of a beam, or between the K-th and (K+1)-th rerank scores, below
1e-5 relative (the GPU's bounds and logits are fp32); such rows must stay
under 0.1%, and the output of every other row within the forward's
tolerance (max-abs 1e-2, mean-abs 1e-3)."""
import numpy as np
import pytest
import torch

from long_context_lm_gb300 import fs
from long_context_lm_gb300.inputs import bf16_values, make_inputs
from oracle import fsb as OB
from oracle import oracle as O
from parity import MAX_ABS, MEAN_ABS, sample_rows, to_device

pytestmark = pytest.mark.gpu
TIE = 1e-5


def _params(**kw):
    p = dict(w=512, s=32, K=4, P=64, W=8, Bq=128, rope_base=10000.0, rms_eps=1e-6, mode=2,
             beam=16, tau=0.0)
    p.update(kw)
    return p


def _setup(B, H, N, seed, sigma_ln=0.8, needles="none", n_needles=0):
    inp = make_inputs(B, H, N, seed=seed, sigma_ln=sigma_ln, needles=needles, n_needles=n_needles)
    q, k, v = [bf16_values(t).reshape(B * H, N, 64).numpy().astype(np.float64)
               for t in (inp.q, inp.k, inp.v)]
    kbar, amax = O.cells(k.astype(np.float32), s=32)
    return inp, q, k, v, kbar, amax


def _compare_sel(gsel, inp, q, k, kbar, amax, params, rows):
    H = inp.q.shape[1]
    ties = 0
    refs = {}
    for bh in range(q.shape[0]):
        h = bh % H
        sel, gap, lgap = OB.fsb_select(q[bh], k[bh], kbar[bh], amax[bh], float(inp.lam[h]),
                                       float(inp.sigma[h]), params["tau"], rows,
                                       K=params["K"], beam=params["beam"])
        refs[bh] = sel
        for i, n in enumerate(rows):
            a = sorted(int(c) for c in gsel[bh, n] if c >= 0)
            b = sorted(int(c) for c in sel[i] if c >= 0)
            if a != b:
                assert min(gap[i], lgap[i]) < TIE, (bh, n, a, b, gap[i], lgap[i])
                ties += 1
    assert ties <= 1e-3 * q.shape[0] * len(rows) + 1, ties
    return refs, ties


@pytest.mark.parametrize("B,H,N,tau,beam,seed", [
    (1, 2, 2048, 0.0, 16, 0),     # every cell in both forests
    (1, 2, 4096, 30.0, 16, 1),    # a strict norm threshold: a smaller second forest
    (2, 1, 3072, 20.0, 4, 2),     # a narrow beam
    (1, 2, 8192, 25.0, 16, 3),    # deeper forests (256 cells)
])
def test_fsb_select_matches_oracle(B, H, N, tau, beam, seed):
    params = _params(tau=tau, beam=beam)
    inp, q, k, v, kbar, amax = _setup(B, H, N, seed)
    d = to_device(inp)
    kb, am = fs.fs_cell_summarize(d["k"])
    sel = fs.fs_fsb_select(d["q"], d["k"], kb, am, d["lam"], d["sigma"], params)
    gsel = sel.cpu().numpy().reshape(B * H, N, -1)
    rows = sample_rows(N, n_blocks=12, per_block=10, seed=seed)
    _, ties = _compare_sel(gsel, inp, q, k, kbar, amax, params, rows)
    print("near ties", ties)


def test_fsb_forward_matches_oracle_and_finds_needles():
    # needles as in the 256k workload: a key 12x a later query, a norm well
    # above the threshold tau, so its cell sits in the second forest and its
    # node's largest norm leads the bound
    B, H, N = 1, 4, 8192
    params = _params(tau=25.0)
    inp, q, k, v, kbar, amax = _setup(B, H, N, 7, sigma_ln=0.5, needles="deep", n_needles=1)
    d = to_device(inp)
    ws = torch.empty(fs.fs_workspace_bytes(B, H, N, 64, params), device="cuda", dtype=torch.uint8)
    out = fs.fs_attention_fwd(d["q"], d["k"], d["v"], d["lam"], d["sigma"], d["mix"], params,
                              ws=ws)
    fs.fs_check_status(ws)
    gout = out.cpu().numpy().reshape(B * H, N, 64)
    gsel = fs.fs_workspace_view(ws, B, H, N, 64, params)["sel"].cpu().numpy().reshape(B * H, N, -1)
    rows = np.unique(np.concatenate([sample_rows(N, 10, 8, seed=7),
                                     np.asarray([j for (_, _, _, j) in inp.needles])]))
    refs, _ = _compare_sel(gsel, inp, q, k, kbar, amax, params, rows)
    # window branch from the oracle forward; long branch from the oracle's
    # readout of the GPU's own selection (near-tie rows included), then the mix
    win = O.forward(q.astype(np.float32), k.astype(np.float32), v.astype(np.float32), H,
                    inp.lam.numpy(), inp.sigma.numpy(), inp.mix.numpy(), rows=rows,
                    params=dict(params, mode=1))["o_win"]
    err = []
    for bh in range(B * H):
        h = bh % H
        for i, n in enumerate(rows):
            ol = O.readout(q[bh].astype(np.float32), k[bh].astype(np.float32),
                           v[bh].astype(np.float32), int(n), gsel[bh, n].tolist())
            ref = win[bh, i] + float(inp.mix[h]) * ol
            err.append(np.abs(gout[bh, n] - ref))
    err = np.asarray(err)
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (err.max(), err.mean())
    # planted needles: the needle's cell is selected by its query
    hits = [p // 32 in gsel[b * H + h, j].tolist() for (b, h, p, j) in inp.needles]
    assert all(hits), (hits, inp.needles)
