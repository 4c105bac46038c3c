"""fs_attention_fwd inside a CUDA graph (GPU only).

The forward is six kernel launches on the caller's stream, with no
host synchronisation, so stream capture records it whole.  A captured
forward must replay to the eager result bit for bit, and recompute when the
inputs in its buffers change.  A warm-up call precedes the capture: the
first call looks up the driver entry point that encodes the TMA tensor maps."""
import pytest
import torch

from long_context_lm_gb300 import fs
from long_context_lm_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


def test_forward_in_cuda_graph_matches_eager():
    B, H, N = 1, 4, 4096
    inp = make_inputs(B, H, N, seed=9, sigma_ln=0.8)
    q, k, v = (t.cuda() for t in (inp.q, inp.k, inp.v))
    lam, sigma, mix = (t.cuda() for t in (inp.lam, inp.sigma, inp.mix))
    params = fs.fs_default_params()
    ws = torch.empty(fs.fs_workspace_bytes(B, H, N, 64, params, fs.FS_BF16), device="cuda",
                     dtype=torch.uint8)
    ref = fs.fs_attention_fwd(q, k, v, lam, sigma, mix, params, ws=ws).clone()

    out = torch.empty_like(ref)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up on the stream the capture will use
        fs.fs_attention_fwd(q, k, v, lam, sigma, mix, params, out=out, ws=ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fs.fs_attention_fwd(q, k, v, lam, sigma, mix, params, out=out, ws=ws)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)

    # new values in the captured buffers: the replay recomputes everything
    k.copy_(torch.roll(k, shifts=1, dims=2))
    v.mul_(0.5)
    ref2 = fs.fs_attention_fwd(q, k, v, lam, sigma, mix, params).clone()
    g.replay()
    torch.cuda.synchronize()
    assert not torch.equal(ref2, ref)
    assert torch.equal(out, ref2)
