"""Device-side error reporting (GPU only), without faulting the GPU.

* A bounded wait that runs out: the self-test kernel waits on an mbarrier
  that nothing completes; after its limit it records FS_ERR_TIMEOUT in the
  workspace header and returns, and the context stays usable.
* A value of v past the fp16 range of the window's P.V product is reported
  as FS_ERR_RANGE by the next status check."""
import pytest
import torch

from long_context_lm_gb300 import fs
from long_context_lm_gb300.inputs import make_inputs
from parity import to_device

pytestmark = pytest.mark.gpu
PAGE = dict(w=512, s=32, K=4, P=64, W=8, Bq=128, rope_base=10000.0, rms_eps=1e-6, mode=0)


def test_bounded_wait_reports_timeout_and_context_survives():
    ws = torch.zeros(256, device="cuda", dtype=torch.uint8)
    fs.fs_selftest_wait_timeout(ws)
    with pytest.raises(fs.FSError) as e:
        fs.fs_check_status(ws)
    assert e.value.status == fs.FS_ERR_TIMEOUT
    # the device still works: a normal forward afterwards checks clean
    inp = make_inputs(1, 2, 1024, seed=3)
    d = to_device(inp)
    B, H, N, dd = inp.q.shape
    ws2 = torch.empty(fs.fs_workspace_bytes(B, H, N, dd, PAGE), device="cuda", dtype=torch.uint8)
    out = fs.fs_attention_fwd(d["q"], d["k"], d["v"], d["lam"], d["sigma"], d["mix"], PAGE, ws=ws2)
    fs.fs_check_status(ws2)
    assert torch.isfinite(out).all()


def test_value_past_fp16_range_is_reported():
    inp = make_inputs(1, 1, 1024, seed=4)
    inp.v[0, 0, 700, 5] = 1.0e5  # finite in bf16, past the fp16 range
    d = to_device(inp)
    B, H, N, dd = inp.q.shape
    ws = torch.empty(fs.fs_workspace_bytes(B, H, N, dd, PAGE), device="cuda", dtype=torch.uint8)
    fs.fs_attention_fwd(d["q"], d["k"], d["v"], d["lam"], d["sigma"], d["mix"], PAGE, ws=ws)
    with pytest.raises(fs.FSError) as e:
        fs.fs_check_status(ws)
    assert e.value.status == fs.FS_ERR_RANGE
    # a clean input on the same workspace clears it again
    d["v"][0, 0, 700, 5] = 0.5
    fs.fs_attention_fwd(d["q"], d["k"], d["v"], d["lam"], d["sigma"], d["mix"], PAGE, ws=ws)
    fs.fs_check_status(ws)
