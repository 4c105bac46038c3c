"""fs_decode_step against the fp64 oracle (GPU only).

A run of decode steps must reproduce, token by token, rows of the full
forward computed by the oracle on the same sequence (outputs within the
tolerance, selections exact up to near ties), and must leave the state as the
prefill kernels would build it: closed cells' summaries bit for bit, and the
pool advanced at a block start exactly as fs_prune_cells computes it."""
import numpy as np
import pytest
import torch

from long_context_lm_gb300 import fs
from long_context_lm_gb300.inputs import make_inputs
from parity import compare_forward, oracle_rows, to_device

pytestmark = pytest.mark.gpu
PAGE = dict(w=512, s=32, K=4, P=64, W=8, Bq=128, rope_base=10000.0, rms_eps=1e-6, mode=0)


def _prefix_state(d, N, t0, params):
    """Caller state before token t0: history rows < t0 (later rows poisoned),
    summaries of cells < t0/32 (later ones NaN), pool of block (t0-1)/128."""
    B, H = d["k"].shape[:2]
    kc = d["k"].clone()
    vc = d["v"].clone()
    kc[:, :, t0:] = float("nan")
    vc[:, :, t0:] = float("nan")
    kbar_full, amax_full = fs.fs_cell_summarize(d["k"])
    kbar = kbar_full.clone()
    amax = amax_full.clone()
    kbar[:, :, t0 // 32:] = float("nan")
    amax[:, :, t0 // 32:] = float("nan")
    cap = params["P"] + params["W"]
    if t0 == 0:
        pool = torch.full((B, H, cap), -1, device="cuda", dtype=torch.int32)
        count = torch.zeros((B, H), device="cuda", dtype=torch.int32)
    else:
        full_pool, full_count = fs.fs_prune_cells(amax_full, N, params)
        blk = (t0 - 1) // 128
        pool = full_pool[:, :, blk].contiguous()
        count = full_count[:, :, blk].contiguous()
    return dict(k_cache=kc, v_cache=vc, kbar=kbar, amax=amax, pool=pool, pool_count=count)


def _run(inp, t0, t1, params):
    d = to_device(inp)
    B, H, N, dd = inp.q.shape
    st = _prefix_state(d, N, t0, params)
    out = np.zeros((B * H, N, dd), np.float32)
    sel = np.full((B * H, N, params["K"]), -1, np.int32)
    s_t = torch.empty((B, H, params["K"]), device="cuda", dtype=torch.int32)
    for t in range(t0, t1):
        o = fs.fs_decode_step(d["q"][:, :, t].contiguous(), d["k"][:, :, t].contiguous(),
                              d["v"][:, :, t].contiguous(), t, st, d["lam"], d["sigma"],
                              d["mix"], params, sel=s_t)
        out[:, t] = o.cpu().numpy().reshape(B * H, dd)
        sel[:, t] = s_t.cpu().numpy().reshape(B * H, -1)
    torch.cuda.synchronize()
    return d, st, out, sel


@pytest.mark.parametrize("N,t0,t1,H,sigma_ln", [
    (4352, 4096 - 40, 4096 + 40, 3, 0.8),
    (384, 0, 300, 2, 0.8),
    # the benchmark's decode context: 16 heads, t around 65536 (a block start,
    # where the pool advances), lognormal spread of the 64k workload
    (65536 + 128, 65536 - 40, 65536 + 40, 16, 0.5),
])
def test_decode_rows_match_oracle_and_state(N, t0, t1, H, sigma_ln):
    params = dict(PAGE)
    inp = make_inputs(1, H, N, seed=N + t0, sigma_ln=sigma_ln,
                      needles="uniform" if N > 2048 else "none", n_needles=4)
    d, st, out, sel = _run(inp, t0, t1, params)
    rows = np.arange(t0, t1)
    compare_forward(inp, params, rows, out, sel)
    # state: every cell closed during the run, bit for bit as the prefill writes it
    kbar_ref, amax_ref = fs.fs_cell_summarize(d["k"])
    c0, c1 = t0 // 32, t1 // 32
    assert torch.equal(st["amax"][:, :, c0:c1], amax_ref[:, :, c0:c1])
    assert torch.equal(st["kbar"][:, :, c0:c1], kbar_ref[:, :, c0:c1])
    # pool: the block of token t1-1, as fs_prune_cells builds it
    pool_ref, count_ref = fs.fs_prune_cells(amax_ref, N, params)
    blk = (t1 - 1) // 128
    assert torch.equal(st["pool_count"], count_ref[:, :, blk])
    assert torch.equal(st["pool"], pool_ref[:, :, blk])
    # history rows written by the steps
    assert torch.equal(st["k_cache"][:, :, t0:t1], d["k"][:, :, t0:t1])
    assert torch.equal(st["v_cache"][:, :, t0:t1], d["v"][:, :, t0:t1])


def test_decode_small_window_and_k():
    params = dict(PAGE, w=64, K=2, P=8, W=2)
    N, t0, t1 = 1024, 600, 700
    inp = make_inputs(1, 2, N, seed=5, sigma_ln=0.8)
    _, _, out, sel = _run(inp, t0, t1, params)
    compare_forward(inp, params, np.arange(t0, t1), out, sel)


def test_decode_rejects_bad_arguments():
    inp = make_inputs(1, 1, 256, seed=1)
    d = to_device(inp)
    st = _prefix_state(d, 256, 0, PAGE)
    q = d["q"][:, :, 0].contiguous()
    with pytest.raises(fs.FSError):  # t past the capacity
        fs.fs_decode_step(q, q, q, 256, st, d["lam"], d["sigma"], d["mix"], PAGE)
    with pytest.raises(fs.FSError):  # FS mode keeps no bounded pool
        fs.fs_decode_step(q, q, q, 0, st, d["lam"], d["sigma"], d["mix"], dict(PAGE, mode=1))
