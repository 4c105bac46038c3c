"""The forward's one pass over k and v (rotated keys, fp16 values and cell
summaries together) against the stand-alone kernels (GPU only), bit for bit.

- Cell summaries: the forward's workspace holds kbar and a_c equal to what
  fs_cell_summarize computes from the same keys.
- Rotated keys and fp16 values: with every mix weight 0 the forward's output
  is its window branch alone (0 times a finite long-branch value adds 0), so
  it equals fs_window_attn, whose operands come from the stand-alone prep
  kernel; any difference in the prepared operands would show."""
import pytest
import torch

from long_context_lm_gb300 import fs
from long_context_lm_gb300.inputs import make_inputs
from parity import to_device

pytestmark = pytest.mark.gpu
PAGE = dict(w=512, s=32, K=4, P=64, W=8, Bq=128, rope_base=10000.0, rms_eps=1e-6, mode=0)


@pytest.mark.parametrize("B,H,N,sig", [(1, 3, 4096, 0.8), (2, 2, 8192 + 128, 0.5)])
def test_fused_prep_matches_standalone_kernels(B, H, N, sig):
    inp = make_inputs(B, H, N, seed=N + H, sigma_ln=sig, needles="uniform", n_needles=2)
    d = to_device(inp)
    params = fs.fs_default_params(**PAGE)
    ws = torch.empty(fs.fs_workspace_bytes(B, H, N, 64, params), device="cuda", dtype=torch.uint8)
    zero_mix = torch.zeros_like(d["mix"])
    out = fs.fs_attention_fwd(d["q"], d["k"], d["v"], d["lam"], d["sigma"], zero_mix, params, ws=ws)
    view = fs.fs_workspace_view(ws, B, H, N, 64, params)
    kbar, amax = fs.fs_cell_summarize(d["k"])
    win = fs.fs_window_attn(d["q"], d["k"], d["v"], params=params)
    torch.cuda.synchronize()
    assert torch.equal(view["kbar"], kbar)
    assert torch.equal(view["amax"], amax)
    assert torch.equal(out, win)
