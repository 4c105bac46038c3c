"""Decoding from the bounded FS-L state against the fp64 oracle (GPU only).

A run of fs_decode_step calls must reproduce, token by token, rows of the
full forward computed by the oracle on the same sequence (outputs within the
tolerance, selections exact up to near ties), whether the state starts empty
or is built from a prefill (fs_decode_state_init).  The state's closed-cell
summaries must equal fs_cell_summarize bit for bit, the two starts must give
bit-identical outputs, and the state never changes size."""
import numpy as np
import pytest
import torch

from long_context_lm_gb300 import fs
from long_context_lm_gb300.inputs import make_inputs
from parity import compare_forward, to_device

pytestmark = pytest.mark.gpu
PAGE = dict(w=512, s=32, K=4, P=64, W=8, Bq=128, rope_base=10000.0, rms_eps=1e-6, mode=0)


def _init_state(d, N, N0, params):
    """State after the first N0 tokens, built from the prefill kernels."""
    B, H = d["k"].shape[:2]
    if N0 == 0:
        return fs.fs_decode_state_init(B, H, params, N0=0)
    kbar, amax = fs.fs_cell_summarize(d["k"])
    pool, count = fs.fs_prune_cells(amax, N, params)
    return fs.fs_decode_state_init(B, H, params, k=d["k"], v=d["v"], kbar=kbar, amax=amax,
                                   pool=pool, pool_count=count, N0=N0)


def _decode(d, state, t0, t1, params):
    B, H, N, dd = d["q"].shape
    out = np.zeros((B * H, N, dd), np.float32)
    sel = np.full((B * H, N, params["K"]), -1, np.int32)
    o = torch.empty((B, H, dd), device="cuda", dtype=torch.float32)
    s_t = torch.empty((B, H, params["K"]), device="cuda", dtype=torch.int32)
    outs, sels = [], []
    for t in range(t0, t1):
        fs.fs_decode_step(d["q"][:, :, t].contiguous(), d["k"][:, :, t].contiguous(),
                          d["v"][:, :, t].contiguous(), t, state, d["lam"], d["sigma"], d["mix"],
                          params, out=o, sel=s_t)
        outs.append(o.clone())
        sels.append(s_t.clone())
    fs.fs_check_status(state)
    torch.cuda.synchronize()
    if outs:
        out[:, t0:t1] = torch.stack(outs, 2).cpu().numpy().reshape(B * H, t1 - t0, dd)
        sel[:, t0:t1] = torch.stack(sels, 2).cpu().numpy().reshape(B * H, t1 - t0, -1)
    return out, sel


def _check_summaries(d, state, params):
    # every closed cell the state holds carries the prefill's summary, bit for bit
    B, H = d["k"].shape[:2]
    kbar, amax = fs.fs_cell_summarize(d["k"])
    view = fs.fs_decode_state_view(state, B, H, params)
    kb = kbar.reshape(B * H, -1, 64)
    am = amax.reshape(B * H, -1)
    n = 0
    for bh in range(B * H):
        cells = view["cell"][bh]
        for sl in torch.nonzero(cells >= 0).flatten().tolist():
            c = int(cells[sl])
            assert torch.equal(view["kbar"][bh, sl], kb[bh, c]), (bh, sl, c)
            assert torch.equal(view["amax"][bh, sl], am[bh, c]), (bh, sl, c)
            n += 1
    return n


@pytest.mark.parametrize("N,H,params", [
    (1024, 2, PAGE),
    (1024, 2, dict(PAGE, w=64, K=2, P=8, W=2)),   # heavy pruning, pool turnover
])
def test_decode_from_empty_state_matches_oracle(N, H, params):
    inp = make_inputs(1, H, N, seed=N + H, sigma_ln=0.8)
    d = to_device(inp)
    state = _init_state(d, N, 0, params)
    out, sel = _decode(d, state, 0, N, params)
    compare_forward(inp, params, np.arange(N), out, sel)
    assert _check_summaries(d, state, params) > 0


@pytest.mark.parametrize("N0", [1, 31, 32, 127, 128, 129, 640, 2000])
def test_decode_from_prefix_matches_stream_from_empty(N0):
    # the state built from a prefill equals, in what it computes, the state
    # reached by decoding every token from an empty one: outputs bit for bit
    N, H, params = 2304, 2, dict(PAGE, P=16, W=4)
    inp = make_inputs(1, H, N, seed=N0, sigma_ln=0.8)
    d = to_device(inp)
    t1 = min(N, N0 + 160)
    ref_out, ref_sel = _decode(d, _init_state(d, N, 0, params), 0, t1, params)
    state = _init_state(d, N, N0, params)
    out, sel = _decode(d, state, N0, t1, params)
    np.testing.assert_array_equal(sel[:, N0:t1], ref_sel[:, N0:t1])
    np.testing.assert_array_equal(out[:, N0:t1], ref_out[:, N0:t1])
    compare_forward(inp, params, np.arange(N0, t1), out, sel)
    _check_summaries(d, state, params)


@pytest.mark.parametrize("N,t0,t1,H,sigma_ln", [
    (4352, 4096 - 40, 4096 + 40, 3, 0.8),
    # the benchmark's decode context: 16 heads, t around 65536 (a block start,
    # where the pool advances), lognormal spread of the 64k workload
    (65536 + 128, 65536 - 40, 65536 + 40, 16, 0.5),
])
def test_decode_from_prefill_matches_oracle(N, t0, t1, H, sigma_ln):
    params = dict(PAGE)
    inp = make_inputs(1, H, N, seed=N + t0, sigma_ln=sigma_ln, needles="uniform", n_needles=4)
    d = to_device(inp)
    state = _init_state(d, N, t0, params)
    nbytes = state.numel()
    out, sel = _decode(d, state, t0, t1, params)
    compare_forward(inp, params, np.arange(t0, t1), out, sel)
    assert _check_summaries(d, state, params) >= H * (params["P"] + params["W"])
    assert state.numel() == nbytes == fs.fs_decode_state_bytes(1, H, 64, params)


def test_decode_step_at_the_wrong_position_is_reported():
    params = dict(PAGE)
    inp = make_inputs(1, 2, 256, seed=1)
    d = to_device(inp)
    state = _init_state(d, 256, 0, params)
    q = d["q"][:, :, 0].contiguous()
    fs.fs_decode_step(q, q, q, 5, state, d["lam"], d["sigma"], d["mix"], params)  # state is at 0
    with pytest.raises(fs.FSError) as e:
        fs.fs_check_status(state)
    assert e.value.status == fs.FS_ERR_STATE
    # nothing changed: the state still takes token 0
    state2 = _init_state(d, 256, 0, params)
    fs.fs_decode_step(q, q, q, 0, state2, d["lam"], d["sigma"], d["mix"], params)
    with pytest.raises(fs.FSError):  # FS mode keeps no bounded pool
        fs.fs_decode_step(q, q, q, 0, state2, d["lam"], d["sigma"], d["mix"], dict(PAGE, mode=1))
