"""The shared q / k / v projection (RMSNorm + W_q/W_k/W_v, one tcgen05 GEMM)
against the fp64 oracle (GPU only).

Error bound of the kernel, element by element, from its arithmetic (u =
2^-8, the unit roundoff of bf16's 8-bit significand): the gain is folded into
the weights as bf16(w * g) (relative error <= u per weight, none when the gain
is absent), products accumulate in fp32 and the result is rounded once to
bf16 (<= u relative).  So
    |gpu - ref| <= u * |ref| + eps_w * S,   S = sum_i |RMSNorm(x)_i * w_i|,
with eps_w = u with a gain and about 2^-20 (fp32 accumulation) without; the
test allows 1% slack on each term."""
import numpy as np
import pytest
import torch

from long_context_lm_gb300 import fs
from long_context_lm_gb300.inputs import make_prologue_inputs
from oracle.prologue import qkv_prologue, rms_norm

pytestmark = pytest.mark.gpu


def _check(inp, H, q, k, v, rows=None, gain=True):
    x = inp.x.float().numpy().astype(np.float64)
    w = inp.w_qkv.float().numpy().astype(np.float64)
    g = inp.gain.numpy().astype(np.float64) if gain else np.ones(x.shape[-1])
    if rows is not None:
        x = x[:, rows]
    ref = qkv_prologue(x, g, w, H, 64, eps=1e-6)
    xn = rms_norm(x, g, 1e-6)
    S = np.abs(xn) @ np.abs(w).T  # [B, R, 3*H*64]
    B, R = x.shape[:2]
    S = S.reshape(B, R, 3, H, 64).transpose(2, 0, 3, 1, 4)
    u = 2.0 ** -8
    eps_w = u if gain else 2.0 ** -20
    worst = 0.0
    for which, got in enumerate((q, k, v)):
        got = got.float().cpu().numpy().astype(np.float64)
        if rows is not None:
            got = got[:, :, rows]
        err = np.abs(got - ref[which])
        bound = 1.01 * (u * np.abs(ref[which]) + eps_w * S[which]) + 1e-7
        assert np.all(err <= bound), (which, float((err / bound).max()))
        worst = max(worst, float((err / bound).max()))
    return worst


@pytest.mark.parametrize("B,N,D,H,gain", [
    (1, 128, 64, 1, True),      # one tile
    (2, 256, 1024, 16, True),   # the layer shape, several tiles per SM row
    (1, 384, 128, 3, False),    # odd head count: tiles of three heads of q, k, v
    (3, 640, 256, 5, True),     # more tiles than SMs, ragged last wave
])
def test_prologue_matches_oracle(B, N, D, H, gain):
    inp = make_prologue_inputs(B, N, D, H, seed=B + N + D + H, gain="random" if gain else "ones")
    q, k, v = fs.fs_qkv_prologue(inp.x.cuda(), inp.w_qkv.cuda(), H,
                                 gain=inp.gain.cuda() if gain else None)
    torch.cuda.synchronize()
    print(_check(inp, H, q, k, v, gain=gain))


def test_prologue_full_size_sampled_rows():
    # the benchmark's layer: 64k tokens, d_model 1024, 16 heads; rows sampled
    B, N, D, H = 1, 65536, 1024, 16
    inp = make_prologue_inputs(B, N, D, H, seed=3)
    q, k, v = fs.fs_qkv_prologue(inp.x.cuda(), inp.w_qkv.cuda(), H, gain=inp.gain.cuda())
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, 127, 128, N - 1], rng.integers(0, N, 200)]))
    print(_check(inp, H, q, k, v, rows=rows))


def test_prologue_repeat_calls_are_identical_and_bad_arguments_rejected():
    inp = make_prologue_inputs(1, 256, 128, 2, seed=7)
    x, w, g = inp.x.cuda(), inp.w_qkv.cuda(), inp.gain.cuda()
    a = fs.fs_qkv_prologue(x, w, 2, gain=g)
    b = fs.fs_qkv_prologue(x, w, 2, gain=g)
    for u, v in zip(a, b):
        assert torch.equal(u, v)
    assert fs.fs_qkv_workspace_bytes(1, 100, 128, 2) == 0   # N not a multiple of 128
    assert fs.fs_qkv_workspace_bytes(1, 256, 100, 2) == 0   # D not a multiple of 64
    with pytest.raises(ValueError):
        fs.fs_qkv_prologue(x, w, 3, gain=g)                 # weight rows do not match H
