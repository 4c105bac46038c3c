"""Pins of the q / k / v projection oracle (oracle/prologue.py) against things
other than itself: PyTorch's RMSNorm and linear in float64 (library
routines), a per-element loop on a tiny case (the head and q/k/v index
mapping), the scale invariance of RMSNorm, and an identity projection."""
import numpy as np
import pytest
import torch

from oracle.prologue import qkv_prologue, rms_norm


def _inputs(B, N, D, H, d, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B, N, D)) * rng.lognormal(0, 0.5, size=(B, N, 1))
    g = rng.uniform(0.5, 1.5, size=D)
    w = rng.standard_normal((3 * H * d, D)) / np.sqrt(D)
    return x, g, w


def test_matches_torch_rms_norm_and_linear():
    B, N, D, H, d = 2, 7, 48, 3, 16
    x, g, w = _inputs(B, N, D, H, d, 0)
    q, k, v = qkv_prologue(x, g, w, H, d, eps=1e-6)
    xt = torch.from_numpy(x)
    xn = torch.nn.functional.rms_norm(xt, (D,), weight=torch.from_numpy(g), eps=1e-6)
    y = torch.nn.functional.linear(xn, torch.from_numpy(w)).numpy()  # [B, N, 3*H*d]
    for which, got in enumerate((q, k, v)):
        want = y[..., which * H * d:(which + 1) * H * d].reshape(B, N, H, d).transpose(0, 2, 1, 3)
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_index_mapping_by_loops():
    B, N, D, H, d = 1, 3, 5, 2, 3
    x, g, w = _inputs(B, N, D, H, d, 1)
    q, k, v = qkv_prologue(x, g, w, H, d, eps=0.0)
    for b in range(B):
        for n in range(N):
            ms = sum(float(x[b, n, i]) ** 2 for i in range(D)) / D
            xn = [float(x[b, n, i]) / ms ** 0.5 * float(g[i]) for i in range(D)]
            for which, t in enumerate((q, k, v)):
                for h in range(H):
                    for j in range(d):
                        row = which * H * d + h * d + j
                        ref = sum(xn[i] * float(w[row, i]) for i in range(D))
                        assert abs(t[b, h, n, j] - ref) < 1e-12


def test_rms_norm_is_scale_invariant_and_identity_projection():
    B, N, D, H, d = 1, 4, 32, 2, 16
    x, g, w = _inputs(B, N, D, H, d, 2)
    a = qkv_prologue(x, g, w, H, d, eps=0.0)
    b = qkv_prologue(x * 37.5, g, w, H, d, eps=0.0)
    for u, v in zip(a, b):
        np.testing.assert_allclose(u, v, rtol=1e-12, atol=1e-13)
    # identity projection (H*d == D): q is RMSNorm(x) split into heads
    eye = np.concatenate([np.eye(D)] * 3)
    q, _, _ = qkv_prologue(x, np.ones(D), eye, H, d, eps=0.0)
    xn = x / np.sqrt(np.mean(x * x, -1, keepdims=True))
    np.testing.assert_allclose(q, xn.reshape(B, N, H, d).transpose(0, 2, 1, 3), rtol=1e-12)
    # unit RMS after the norm (gain 1, eps 0)
    np.testing.assert_allclose(np.mean(rms_norm(x, np.ones(D), 0.0) ** 2, -1), 1.0, rtol=1e-12)
