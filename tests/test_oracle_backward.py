"""Pins of the oracle's backward pass (CPU).

The backward (oracle.backward) holds each row's pool and selection fixed: the
pages state that the hard top-P / top-K indices carry no gradient and that
sigma_h and lambda_h are fixed ("FreeSolo: Linear-time Sparse Attention with
Zero-Shot Length Extrapolation": paper.rainbus.top summary, 方法步骤详情 and
局限与改进; ai.info summary, "Methodology in Plain English").  Two checks
that share none of its formulas:

- central finite differences of L = sum(g * out) through the oracle's own
  forward (pinned elsewhere), with perturbations exact in float32, on
  coordinates whose perturbation leaves every selection unchanged;
- PyTorch autograd (float64) through a dense formulation written here: RoPE
  as complex multiplication, a banded causal mask for the window, a token
  mask from the selection for the long branch, RMSNorm and the mix."""
import numpy as np
import pytest
import torch

from oracle import oracle

TINY = dict(w=24, s=8, K=2, P=4, W=2, Bq=32, rope_base=10000.0, rms_eps=1e-6, mode=0)


def _inputs(BH, N, d, seed, sigma_ln=0.5):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((BH, N, d)).astype(np.float32)
    k = (rng.standard_normal((BH, N, d)) * np.exp(sigma_ln * rng.standard_normal((BH, N, 1))))
    k = k.astype(np.float32)
    v = rng.standard_normal((BH, N, d)).astype(np.float32)
    g = rng.standard_normal((BH, N, d))
    return q, k, v, g


def _loss_and_sel(q, k, v, H, lam, sig, mix, g, params):
    r = oracle.forward(q, k, v, H, lam, sig, mix, params=params, want_branches=False)
    return float(np.sum(g * r["out"])), r["sel"]


@pytest.mark.parametrize("mode", [0, 1])
def test_backward_matches_central_differences(mode):
    params = dict(TINY, mode=mode)
    BH, H, N, d = 2, 2, 256, 8
    q, k, v, g = _inputs(BH, N, d, seed=3 + mode)
    lam, sig, mix = np.array([1.0, 0.7]), np.array([4.0, 4.0]), np.array([0.6, 0.35])
    grads = oracle.backward(q, k, v, H, lam, sig, mix, g, params)
    _, sel0 = _loss_and_sel(q, k, v, H, lam, sig, mix, g, params)
    rng = np.random.default_rng(11)
    h = 2.0 ** -12  # x +- h is exact in float32 for |x| < 2048
    checked = 0
    for name, arr in (("dq", q), ("dk", k), ("dv", v)):
        for _ in range(40):
            idx = (int(rng.integers(BH)), int(rng.integers(N)), int(rng.integers(d)))
            xs = []
            for sgn in (1.0, -1.0):
                x = arr.copy()
                x[idx] = np.float32(x[idx] + sgn * h)
                assert float(x[idx]) == float(arr[idx]) + sgn * h
                xs.append(x)
            args = [[q, k, v] for _ in range(2)]
            pos = {"dq": 0, "dk": 1, "dv": 2}[name]
            for a, x in zip(args, xs):
                a[pos] = x
            lp, sp = _loss_and_sel(*args[0], H, lam, sig, mix, g, params)
            lm, sm = _loss_and_sel(*args[1], H, lam, sig, mix, g, params)
            if not (np.array_equal(sp, sel0) and np.array_equal(sm, sel0)):
                continue  # the perturbation moved a hard index: no derivative there
            fd = (lp - lm) / (2 * h)
            an = grads[name][idx]
            assert abs(fd - an) <= 1e-6 + 1e-6 * abs(an), (name, idx, fd, an)
            checked += 1
    assert checked >= 100
    for hh in range(H):  # the mix weight enters linearly
        mp, mm = mix.copy(), mix.copy()
        mp[hh] += 1e-3
        mm[hh] -= 1e-3
        fd = (_loss_and_sel(q, k, v, H, lam, sig, mp, g, params)[0]
              - _loss_and_sel(q, k, v, H, lam, sig, mm, g, params)[0]) / 2e-3
        assert abs(fd - grads["dmix"][hh]) <= 1e-8 * max(1.0, abs(fd))


def _rope(x, base):
    N, d = x.shape[-2], x.shape[-1]
    half = d // 2
    theta = base ** (-2.0 * torch.arange(half, dtype=torch.float64) / d)
    ang = torch.arange(N, dtype=torch.float64)[:, None] * theta[None, :]
    z = torch.complex(x[..., :half], x[..., half:]) * torch.polar(torch.ones_like(ang), ang)
    return torch.cat([z.real, z.imag], dim=-1)


def _dense_forward(q, k, v, mix, sel, H, p):
    BH, N, d = q.shape
    s, w, eps = p["s"], p["w"], p["rms_eps"]
    scale = 1.0 / np.sqrt(d)
    n = torch.arange(N)[:, None]
    j = torch.arange(N)[None, :]
    band = (j <= n) & (j >= n - w + 1)
    qr, kr = _rope(q, p["rope_base"]), _rope(k, p["rope_base"])
    sw = (qr @ kr.transpose(-1, -2)) * scale
    o_win = torch.softmax(sw.masked_fill(~band, float("-inf")), dim=-1) @ v
    cell_of = torch.arange(N) // s
    selt = torch.as_tensor(sel, dtype=torch.int64)  # [BH, N, K]
    tok = (selt[..., None] == cell_of[None, None, None, :]).any(dim=2)  # [BH, N, N]
    has = tok.any(dim=-1, keepdim=True)
    sl = (q @ k.transpose(-1, -2)) * scale
    pl = torch.softmax(sl.masked_fill(~tok, float("-inf")).masked_fill(~has, 0.0), dim=-1)
    o = pl @ v
    o_hat = o / torch.sqrt((o * o).mean(dim=-1, keepdim=True) + eps)
    o_hat = torch.where(has, o_hat, torch.zeros_like(o_hat))
    m = mix.repeat(BH // H)[:, None, None]
    return o_win + m * o_hat


@pytest.mark.parametrize("params,BH,H,N,d", [
    (TINY, 2, 2, 256, 8),
    (dict(TINY, mode=1), 2, 1, 256, 16),
    (dict(w=512, s=32, K=4, P=64, W=8, Bq=128, rope_base=10000.0, rms_eps=1e-6, mode=0),
     2, 2, 1024, 64),
])
def test_backward_matches_dense_autograd(params, BH, H, N, d):
    q, k, v, g = _inputs(BH, N, d, seed=N + d)
    lam = np.linspace(0.5, 1.5, H)
    sig = np.full(H, 4.0)
    mix = np.linspace(0.2, 0.9, H)
    ref = oracle.forward(q, k, v, H, lam, sig, mix, params=params, want_branches=False)
    grads = oracle.backward(q, k, v, H, lam, sig, mix, g, params)
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    tm = torch.tensor(mix, dtype=torch.float64, requires_grad=True)
    out = _dense_forward(tq, tk, tv, tm, ref["sel"], H, dict(oracle.DEFAULT_PARAMS, **params))
    np.testing.assert_allclose(out.detach().numpy(), ref["out"], rtol=0, atol=1e-10)
    (out * torch.tensor(g)).sum().backward()
    for name, t in (("dq", tq), ("dk", tk), ("dv", tv)):
        np.testing.assert_allclose(grads[name], t.grad.numpy(), rtol=1e-9, atol=1e-10,
                                   err_msg=name)
    np.testing.assert_allclose(grads["dmix"], tm.grad.numpy(), rtol=1e-10, atol=1e-10)
