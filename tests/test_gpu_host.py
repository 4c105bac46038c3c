"""fs_attention_fwd_host: the forward on host buffers, pipelined over groups
of heads through two device staging slots (GPU only).

Every (batch, head) slice is computed by the same kernels with the same
arithmetic as in fs_attention_fwd, so the outputs must be bit-identical for
any group size, for bf16 and fp32 inputs, with pinned and pageable host
memory.  A device error in any group reaches the call's error word."""
import pytest
import torch

from long_context_lm_gb300 import fs
from long_context_lm_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu
PAGE = dict(w=512, s=32, K=4, P=64, W=8, Bq=128, rope_base=10000.0, rms_eps=1e-6, mode=0)


def _device_ref(inp, params):
    d = [t.cuda() for t in (inp.q, inp.k, inp.v, inp.lam, inp.sigma, inp.mix)]
    return fs.fs_attention_fwd(*d, params).cpu()


@pytest.mark.parametrize("B,H,N,hc,dtype,pinned", [
    (2, 3, 1024, 2, "bf16", True),   # groups of 2 and 1 in each batch row
    (2, 3, 1024, 1, "bf16", True),   # six groups: both slots reused
    (1, 4, 2048, 8, "bf16", False),  # one group, pageable memory
    (1, 2, 512, 1, "fp32", True),    # fp32 staging, rounded in the forward
])
def test_host_forward_matches_device_forward(B, H, N, hc, dtype, pinned):
    inp = make_inputs(B, H, N, seed=B * 10 + H + hc, sigma_ln=0.8, dtype=dtype)
    params = fs.fs_default_params(**PAGE)
    ref = _device_ref(inp, params)
    q, k, v = inp.q.contiguous(), inp.k.contiguous(), inp.v.contiguous()
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    lam, sigma, mix = inp.lam.cuda(), inp.sigma.cuda(), inp.mix.cuda()
    out = torch.full((B, H, N, 64), float("nan"), dtype=torch.float32)
    if pinned:
        out = out.pin_memory()
    ws = torch.empty(fs.fs_host_workspace_bytes(B, H, N, 64, params,
                                                fs.FS_FP32 if dtype == "fp32" else fs.FS_BF16, hc),
                     device="cuda", dtype=torch.uint8)
    for _ in range(2):  # the second call reuses the workspace and the copy streams
        out.fill_(float("nan"))
        fs.fs_attention_fwd_host(q, k, v, lam, sigma, mix, params, out=out, ws=ws,
                                 heads_per_chunk=hc)
        fs.fs_check_status(ws)
        assert torch.equal(out, ref)


def test_host_forward_back_to_back_calls_with_different_inputs():
    # Two calls on one workspace and stream with no synchronisation between
    # them: the second call's loads into the staging slots wait for the first
    # call's forwards and stores, so each output matches its own inputs.
    B, H, N, hc = 1, 4, 2048, 1
    params = fs.fs_default_params(**PAGE)
    inps = [make_inputs(B, H, N, seed=90 + i, sigma_ln=0.8) for i in range(2)]
    refs = [_device_ref(inp, params) for inp in inps]
    assert not torch.equal(refs[0], refs[1])
    lam, sigma, mix = inps[0].lam.cuda(), inps[0].sigma.cuda(), inps[0].mix.cuda()
    host = [[t.contiguous().pin_memory() for t in (inp.q, inp.k, inp.v)] for inp in inps]
    # the second call runs on the first call's per-head parameters
    refs[1] = fs.fs_attention_fwd(*[t.cuda() for t in (inps[1].q, inps[1].k, inps[1].v)],
                                  lam, sigma, mix, params).cpu()
    outs = [torch.full((B, H, N, 64), float("nan")).pin_memory() for _ in range(2)]
    ws = torch.empty(fs.fs_host_workspace_bytes(B, H, N, 64, params, fs.FS_BF16, hc),
                     device="cuda", dtype=torch.uint8)
    torch.cuda.synchronize()
    for rep in range(2):
        for o in outs:
            o.fill_(float("nan"))
        for i in range(2):
            fs.fs_attention_fwd_host(*host[i], lam, sigma, mix, params, out=outs[i], ws=ws,
                                     heads_per_chunk=hc)
        fs.fs_check_status(ws)
        assert torch.equal(outs[0], refs[0])
        assert torch.equal(outs[1], refs[1])


def test_host_forward_reports_a_range_error_of_any_group():
    B, H, N = 1, 3, 1024
    inp = make_inputs(B, H, N, seed=4)
    inp.v[0, 2, 700, 5] = 1.0e5  # last group only: finite in bf16, past the fp16 range
    params = fs.fs_default_params(**PAGE)
    lam, sigma, mix = inp.lam.cuda(), inp.sigma.cuda(), inp.mix.cuda()
    ws = torch.empty(fs.fs_host_workspace_bytes(B, H, N, 64, params, fs.FS_BF16, 1), device="cuda",
                     dtype=torch.uint8)
    fs.fs_attention_fwd_host(inp.q, inp.k, inp.v, lam, sigma, mix, params, ws=ws, heads_per_chunk=1)
    with pytest.raises(fs.FSError) as e:
        fs.fs_check_status(ws)
    assert e.value.status == fs.FS_ERR_RANGE
    inp.v[0, 2, 700, 5] = 0.5
    fs.fs_attention_fwd_host(inp.q, inp.k, inp.v, lam, sigma, mix, params, ws=ws, heads_per_chunk=1)
    fs.fs_check_status(ws)


def test_host_forward_rejects_bad_arguments():
    inp = make_inputs(1, 2, 512, seed=1)
    params = fs.fs_default_params(**PAGE)
    lam, sigma, mix = inp.lam.cuda(), inp.sigma.cuda(), inp.mix.cuda()
    with pytest.raises(ValueError):  # device tensors where host ones are expected
        fs.fs_attention_fwd_host(inp.q.cuda(), inp.k, inp.v, lam, sigma, mix, params)
    assert fs.fs_host_workspace_bytes(1, 2, 512, 64, params, fs.FS_BF16, 0) == 0
