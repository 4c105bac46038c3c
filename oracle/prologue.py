"""Shared q / k / v projection of an FS-L layer: plain numpy, float64.

TEST INFRASTRUCTURE ONLY: the tests and the benchmark's CPU leg call it; the
product path never imports it, and it imports nothing from the product.

"FreeSolo: Linear-time Sparse Attention with Zero-Shot Length Extrapolation"
(paper.rainbus.top summary, 方法步骤详情 ①): the hidden state goes through
RMSNorm and the projections W_q, W_k, W_v, giving the q, k, v that both
branches of every head share.

Reading taken (the pages give no formula): RMSNorm(x) = x / sqrt(mean(x^2) +
eps) * g with a per-channel gain g (an input: trained weights are not
available) and eps = 1e-6; the projections have no bias.  The three weight
matrices are stacked as one [3*H*d, D] matrix w_qkv (rows: q, then k, then v;
inside each, head h holds rows h*d .. h*d + d-1), so q[b, h, n, j] =
sum_i RMSNorm(x)[b, n, i] * w_qkv[h*d + j, i].
"""
from __future__ import annotations

import numpy as np


def rms_norm(x, gain, eps=1e-6):
    """x [..., D] -> x / sqrt(mean(x^2) + eps) * gain, float64."""
    x = np.asarray(x, np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(gain, np.float64)


def qkv_prologue(x, gain, w_qkv, H, d, eps=1e-6):
    """x [B, N, D], gain [D], w_qkv [3*H*d, D] -> q, k, v [B, H, N, d] float64."""
    xn = rms_norm(x, gain, eps)
    y = xn @ np.asarray(w_qkv, np.float64).T  # [B, N, 3*H*d]
    B, N, _ = y.shape
    y = y.reshape(B, N, 3, H, d).transpose(2, 0, 3, 1, 4)
    return y[0], y[1], y[2]
