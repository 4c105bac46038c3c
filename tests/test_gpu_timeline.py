"""The attention kernel's per-CTA timeline (fs_set_attention_timeline) on
GB300: every CTA of a launch records a start and an end, nothing past the
launch's CTAs is written, and with the timeline off a forward writes none."""
import pytest
import torch

from long_context_lm_gb300 import fs
from long_context_lm_gb300.inputs import make_inputs
from parity import to_device

pytestmark = pytest.mark.gpu


def test_timeline_records_every_cta_of_a_forward():
    B, H, N = 1, 2, 4096
    inp = make_inputs(B, H, N, seed=11)
    d = to_device(inp)
    params = fs.fs_default_params()
    nitems = B * H * N // 128
    grid = min(nitems, torch.cuda.get_device_properties(0).multi_processor_count)
    buf = torch.zeros(2 * 512, dtype=torch.int64, device="cuda")
    fs.fs_set_attention_timeline(buf)
    try:
        fs.fs_attention_fwd(d["q"], d["k"], d["v"], d["lam"], d["sigma"], d["mix"], params)
        torch.cuda.synchronize()
    finally:
        fs.fs_set_attention_timeline(None)
    t = buf.view(-1, 2).cpu()
    used = t[:grid]
    assert (used[:, 0] > 0).all() and (used[:, 1] >= used[:, 0]).all()
    assert (t[grid:] == 0).all()
    # the CTAs run at the same time: they all start before any finishes
    assert used[:, 0].max() <= used[:, 1].min()
    # off again: a forward leaves a fresh buffer untouched
    buf.zero_()
    fs.fs_attention_fwd(d["q"], d["k"], d["v"], d["lam"], d["sigma"], d["mix"], params)
    torch.cuda.synchronize()
    assert (buf == 0).all()
