"""The C-ABI library builds, loads and exports every symbol include/fs.h
declares; host-side argument validation works without a GPU (no compute
call reaches CUDA here)."""
import ctypes
import os
import re

import pytest

from long_context_lm_gb300 import fs

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "fs.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fs_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("fs_cell_summarize", "fs_prune_cells", "fs_select_cells", "fs_sparse_readout",
                 "fs_window_attn", "fs_attention_fwd"):
        assert want in names


def test_library_exports_every_declared_symbol():
    L = fs.load()
    for name in declared_functions():
        assert hasattr(L, name), name
    assert set(declared_functions()) == set(fs.SYMBOLS)


def test_default_params_are_the_page_values():
    p = fs.fs_default_params()
    assert (p.w, p.s, p.K, p.P, p.W, p.Bq) == (512, 32, 4, 64, 8, 128)
    assert p.mode == fs.FS_MODE_FSL


def test_host_workspace_bytes():
    # two staging slots, each with q, k, v and out of one group of heads and a
    # forward workspace for that group
    one = fs.fs_host_workspace_bytes(1, 16, 65536, 64, heads_per_chunk=1)
    four = fs.fs_host_workspace_bytes(1, 16, 65536, 64, heads_per_chunk=4)
    grp = 4 * 65536 * 64
    assert four >= 2 * (3 * grp * 2 + grp * 4 + fs.fs_workspace_bytes(1, 4, 65536, 64))
    assert one < four < fs.fs_host_workspace_bytes(1, 16, 65536, 64, heads_per_chunk=16)
    # a group never exceeds H heads; the batch does not change the slot size
    assert fs.fs_host_workspace_bytes(1, 3, 2048, 64, heads_per_chunk=8) == \
        fs.fs_host_workspace_bytes(4, 3, 2048, 64, heads_per_chunk=3)
    assert fs.fs_host_workspace_bytes(1, 16, 4096, 64, heads_per_chunk=0) == 0
    assert fs.fs_host_workspace_bytes(1, 16, 4096 + 1, 64) == 0
    assert fs.fs_host_workspace_bytes(1, 2, 2048, 64, dtype=fs.FS_FP32) > \
        fs.fs_host_workspace_bytes(1, 2, 2048, 64, dtype=fs.FS_BF16)


def test_status_strings():
    assert fs.status_string(0) == "ok"
    assert "invalid" in fs.status_string(1)
    assert fs.status_string(99) == "unknown status"


def test_workspace_bytes_validation():
    assert fs.fs_workspace_bytes(1, 16, 65536, 64) > 0
    assert fs.fs_workspace_bytes(1, 16, 65536 + 1, 64) == 0      # N % Bq
    assert fs.fs_workspace_bytes(1, 16, 65536, 128) == 0         # d unsupported
    assert fs.fs_workspace_bytes(0, 16, 65536, 64) == 0
    assert fs.fs_workspace_bytes(1, 16, 4096, 64, dict(P=65)) == 0
    assert fs.fs_workspace_bytes(1, 16, 4096, 64, dict(K=9)) == 0
    assert fs.fs_workspace_bytes(1, 16, 4096, 64, dict(mode=3)) == 0
    # FS-B: its forests take workspace; beam 1..16
    assert fs.fs_workspace_bytes(1, 16, 4096, 64, dict(mode=2)) > fs.fs_workspace_bytes(1, 16, 4096, 64)
    assert fs.fs_workspace_bytes(1, 16, 4096, 64, dict(mode=2, beam=17)) == 0
    assert fs.fs_workspace_bytes(1, 16, 4096, 64, dict(mode=2, beam=0)) == 0
    small = fs.fs_workspace_bytes(1, 2, 2048, 64, dtype=fs.FS_BF16)
    big = fs.fs_workspace_bytes(1, 2, 2048, 64, dtype=fs.FS_FP32)
    assert big - small >= 3 * 2 * 2048 * 64 * 2


def _fwd_status(**kw):
    L = fs.load()
    p = fs.fs_default_params(**kw.pop("params", {}))
    args = dict(q=1, k=1, v=1, dtype=0, batch=1, H=2, N=2048, d=64, lam=1, sigma=1, mix=1,
                out=1, ws=1, wsb=1 << 40)
    args.update(kw)
    vp = lambda x: None if x is None else ctypes.c_void_p(x)
    return L.fs_attention_fwd(vp(args["q"]), vp(args["k"]), vp(args["v"]), args["dtype"],
                              args["batch"], args["H"], args["N"], args["d"], ctypes.byref(p),
                              vp(args["lam"]), vp(args["sigma"]), vp(args["mix"]),
                              vp(args["out"]), vp(args["ws"]), args["wsb"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), fs.FS_ERR_INVALID_ARG),
    (dict(out=None), fs.FS_ERR_INVALID_ARG),
    (dict(N=2000), fs.FS_ERR_INVALID_ARG),
    (dict(N=0), fs.FS_ERR_INVALID_ARG),
    (dict(d=128), fs.FS_ERR_UNSUPPORTED),
    (dict(dtype=7), fs.FS_ERR_INVALID_ARG),
    (dict(wsb=16), fs.FS_ERR_INVALID_ARG),
    (dict(params=dict(s=16, Bq=128)), fs.FS_ERR_UNSUPPORTED),
    (dict(params=dict(Bq=100)), fs.FS_ERR_INVALID_ARG),
    (dict(params=dict(w=0)), fs.FS_ERR_INVALID_ARG),
])
def test_attention_fwd_rejects_bad_arguments_before_launch(kw, status):
    assert _fwd_status(**kw) == status


def test_decode_state_is_bounded():
    # The decode state holds ((P+W)s + w + Bq + s) key and value rows per
    # (batch, head) plus the cells' summaries and its lists, whatever the
    # position: the size takes no sequence length at all.  Rows are bf16,
    # except the window's keys: fp32, kept rotated by their position.
    p = fs.fs_default_params()
    one = fs.fs_decode_state_bytes(1, 1)
    sixteen = fs.fs_decode_state_bytes(1, 16)
    per_head = (sixteen - one) // 15
    assert fs.fs_decode_state_bytes(2, 8) == sixteen
    rows = (p.P + p.W) * p.s + p.w + p.Bq + p.s
    kv_bytes = rows * 64 * 2 * 2 + p.w * 64 * 2
    nslots = p.P + p.W + p.Bq // p.s + 1
    summaries = nslots * (64 + 2) * 4
    assert kv_bytes <= per_head <= kv_bytes + summaries + 4096
    assert per_head < 850 * 1024  # about 0.83 MB per head at the page values
    # shapes the decode kernel is not built for
    assert fs.fs_decode_state_bytes(1, 1, params=dict(w=1024)) == 0
    assert fs.fs_decode_state_bytes(1, 1, params=dict(mode=1)) == 0


def test_attention_timeline_argument_checks():
    # host-side only: the setter stores the pointer, nothing reaches the GPU
    L = fs.load()
    assert L.fs_set_attention_timeline(None, 5) == fs.FS_ERR_INVALID_ARG
    assert L.fs_set_attention_timeline(ctypes.c_void_p(256), 0) == fs.FS_ERR_INVALID_ARG
    assert L.fs_set_attention_timeline(ctypes.c_void_p(256), -2) == fs.FS_ERR_INVALID_ARG
    assert L.fs_set_attention_timeline(None, 0) == fs.FS_OK
