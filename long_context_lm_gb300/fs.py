"""Thin Python binding of the C-ABI library ``libfs.so`` (``include/fs.h``).

Only argument marshalling happens here: tensors are checked for device,
dtype, shape and contiguity, their device pointers and the current CUDA
stream are handed to the library, and a non-zero status raises ``FSError``.
Every step of the computation runs in the library's CUDA kernels; there is no
CPU fallback, and a missing or unbuildable library raises.

Function names match the C entry points.  Tensors follow the C layouts:
q, k, v ``[batch, H, N, d]`` (bf16, or fp32 for ``fs_attention_fwd`` /
``fs_cell_summarize``); per-head ``lam``, ``sigma``, ``mix`` ``[H]`` fp32.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

(FS_OK, FS_ERR_INVALID_ARG, FS_ERR_UNSUPPORTED, FS_ERR_CUDA, FS_ERR_TIMEOUT, FS_ERR_RANGE,
 FS_ERR_SCRATCH_LIMIT, FS_ERR_STATE) = range(8)
FS_BF16, FS_FP32 = 0, 1
FS_MODE_FSL, FS_MODE_FS, FS_MODE_FSB = 0, 1, 2

SYMBOLS = ["fs_default_params", "fs_status_string", "fs_last_cuda_error", "fs_workspace_bytes",
           "fs_set_attention_timeline",
           "fs_prune_workspace_bytes", "fs_window_workspace_bytes", "fs_cell_summarize",
           "fs_prune_cells", "fs_select_cells", "fs_sparse_readout", "fs_window_attn",
           "fs_attention_fwd", "fs_attention_fwd_traced", "fs_workspace_view", "fs_check_status",
           "fs_prune_static_scratch_bytes", "fs_prune_cells_static", "fs_decode_step",
           "fs_selftest_wait_timeout", "fs_host_workspace_bytes", "fs_attention_fwd_host",
           "fs_window_attn_traced", "fs_decode_state_bytes", "fs_decode_state_init",
           "fs_decode_state_view", "fs_qkv_workspace_bytes", "fs_qkv_prologue",
           "fs_backward_workspace_bytes", "fs_attention_bwd",
           "fs_fsb_workspace_bytes", "fs_fsb_select"]
FS_N_STAGES = 4
STAGE_NAMES = ["cells_prep", "prune", "select", "attention"]


class fs_params(ctypes.Structure):
    _fields_ = [("w", ctypes.c_int), ("s", ctypes.c_int), ("K", ctypes.c_int),
                ("P", ctypes.c_int), ("W", ctypes.c_int), ("Bq", ctypes.c_int),
                ("rope_base", ctypes.c_float), ("rms_eps", ctypes.c_float),
                ("mode", ctypes.c_int), ("beam", ctypes.c_int), ("tau", ctypes.c_float)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class FSError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        msg = f"{where}: {status_string(status)} (status {status})"
        if status == FS_ERR_CUDA:
            msg += ": " + load().fs_last_cuda_error().decode()
        super().__init__(msg)


_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _build.LIB


def load(build_if_stale: bool = True):
    """Load libfs.so (compiling it in-tree first when it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build_if_stale:
            _build.build()
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"{_build.LIB} is missing: build it with "
                               "`python -m long_context_lm_gb300.build`")
        L = ctypes.CDLL(_build.LIB)
        P, I, Z, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
        PP = ctypes.POINTER(fs_params)
        L.fs_default_params.argtypes = [PP]
        L.fs_default_params.restype = None
        L.fs_status_string.argtypes = [I]
        L.fs_status_string.restype = ctypes.c_char_p
        L.fs_last_cuda_error.argtypes = []
        L.fs_last_cuda_error.restype = ctypes.c_char_p
        L.fs_workspace_bytes.argtypes = [I, I, I, I, PP, I]
        L.fs_workspace_bytes.restype = Z
        L.fs_prune_workspace_bytes.argtypes = [I, I, I, PP]
        L.fs_prune_workspace_bytes.restype = Z
        L.fs_window_workspace_bytes.argtypes = [I, I, I, I, PP]
        L.fs_window_workspace_bytes.restype = Z
        L.fs_host_workspace_bytes.argtypes = [I, I, I, I, PP, I, I]
        L.fs_host_workspace_bytes.restype = Z
        L.fs_cell_summarize.argtypes = [P, I, I, I, I, I, I, P, P, P]
        L.fs_prune_cells.argtypes = [P, I, I, I, PP, P, P, P, Z, P]
        L.fs_select_cells.argtypes = [P, I, P, P, P, P, P, P, I, I, I, I, PP, P, P, P]
        L.fs_sparse_readout.argtypes = [P, P, P, I, P, I, I, I, I, PP, P, P]
        L.fs_window_attn.argtypes = [P, P, P, I, P, P, I, I, I, I, PP, P, P, Z, P]
        L.fs_window_attn_traced.argtypes = L.fs_window_attn.argtypes + [P]
        L.fs_attention_fwd.argtypes = [P, P, P, I, I, I, I, I, PP, P, P, P, P, P, Z, P]
        L.fs_attention_fwd_traced.argtypes = L.fs_attention_fwd.argtypes + [P]
        L.fs_attention_fwd_host.argtypes = [P, P, P, I, I, I, I, I, PP, P, P, P, P, I, P, Z, P]
        L.fs_workspace_view.argtypes = [I, I, I, I, PP, I] + [ctypes.POINTER(Z)] * 5
        L.fs_check_status.argtypes = [P, P]
        L.fs_set_attention_timeline.argtypes = [P, I]
        L.fs_selftest_wait_timeout.argtypes = [P, P]
        L.fs_prune_static_scratch_bytes.argtypes = []
        L.fs_prune_static_scratch_bytes.restype = Z
        L.fs_prune_cells_static.argtypes = [P, I, I, I, PP, P, P, P]
        L.fs_decode_state_bytes.argtypes = [I, I, I, PP]
        L.fs_decode_state_bytes.restype = Z
        L.fs_decode_state_view.argtypes = [I, I, I, PP, ctypes.POINTER(Z)]
        L.fs_qkv_workspace_bytes.argtypes = [I, I, I, I]
        L.fs_backward_workspace_bytes.argtypes = [I, I, I, I, PP]
        L.fs_fsb_workspace_bytes.argtypes = [I, I, I, PP]
        L.fs_fsb_workspace_bytes.restype = Z
        L.fs_fsb_select.argtypes = [P, P, P, P, P, P, I, I, I, I, PP, P, P, Z, P]
        L.fs_backward_workspace_bytes.restype = Z
        L.fs_attention_bwd.argtypes = [P, P, P, I, I, I, I, I, PP, P, P, P, P, P, P, P, P, P, Z, P]
        L.fs_qkv_workspace_bytes.restype = Z
        L.fs_qkv_prologue.argtypes = [P, P, P, I, I, I, I, F, P, P, P, P, Z, P]
        L.fs_decode_state_init.argtypes = [P, P, I, P, P, P, P, I, I, I, I, I, PP, P, Z, P]
        L.fs_decode_step.argtypes = [P, P, P, I, I, I, I, I, P, P, P, PP, P, Z, P, P, P]
        for name in SYMBOLS:
            if name not in ("fs_default_params", "fs_status_string", "fs_last_cuda_error",
                            "fs_workspace_bytes", "fs_prune_static_scratch_bytes",
                            "fs_prune_workspace_bytes", "fs_window_workspace_bytes",
                            "fs_host_workspace_bytes", "fs_decode_state_bytes",
                            "fs_qkv_workspace_bytes", "fs_backward_workspace_bytes",
                            "fs_fsb_workspace_bytes"):
                getattr(L, name).restype = I
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return load().fs_status_string(int(status)).decode()


def _check(status, where):
    if status != FS_OK:
        raise FSError(status, where)


def fs_default_params(**overrides) -> fs_params:
    p = fs_params()
    load().fs_default_params(ctypes.byref(p))
    for k, v in overrides.items():
        setattr(p, k, v)
    return p


def _params(params):
    if params is None:
        return fs_default_params()
    if isinstance(params, dict):
        return fs_default_params(**params)
    return params


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t, name, dtypes):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _dtype_code(t):
    return FS_BF16 if t.dtype == torch.bfloat16 else FS_FP32


def _qkv_shape(q):
    if q.dim() != 4:
        raise ValueError("q/k/v must be [batch, H, N, d]")
    return tuple(q.shape)


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------

def fs_workspace_bytes(batch, H, N, d, params=None, dtype=FS_BF16) -> int:
    p = _params(params)
    return load().fs_workspace_bytes(batch, H, N, d, ctypes.byref(p), dtype)


def fs_window_workspace_bytes(batch, H, N, d, params=None) -> int:
    p = _params(params)
    return load().fs_window_workspace_bytes(batch, H, N, d, ctypes.byref(p))


def fs_cell_summarize(k, s=32, kbar=None, amax=None, stream=None):
    L = load()
    _dev(k, "k", (torch.bfloat16, torch.float32))
    B, H, N, d = _qkv_shape(k)
    C = N // s
    kbar = kbar if kbar is not None else torch.empty((B, H, C, d), device=k.device, dtype=torch.float32)
    amax = amax if amax is not None else torch.empty((B, H, C), device=k.device, dtype=torch.float32)
    _dev(kbar, "kbar", (torch.float32,))
    _dev(amax, "amax", (torch.float32,))
    _check(L.fs_cell_summarize(_ptr(k), _dtype_code(k), B, H, N, d, s, _ptr(kbar), _ptr(amax),
                               _stream(stream)), "fs_cell_summarize")
    return kbar, amax


def fs_prune_cells(amax, N, params=None, stream=None):
    L = load()
    p = _params(params)
    _dev(amax, "amax", (torch.float32,))
    B, H, C = amax.shape
    nblk = N // p.Bq
    pool = torch.empty((B, H, nblk, p.P + p.W), device=amax.device, dtype=torch.int32)
    count = torch.empty((B, H, nblk), device=amax.device, dtype=torch.int32)
    wsb = L.fs_prune_workspace_bytes(B, H, N, ctypes.byref(p))
    if wsb == 0:
        raise FSError(FS_ERR_INVALID_ARG, "fs_prune_workspace_bytes")
    ws = torch.empty(wsb, device=amax.device, dtype=torch.uint8)
    _check(L.fs_prune_cells(_ptr(amax), B, H, N, ctypes.byref(p), _ptr(pool), _ptr(count),
                            _ptr(ws), wsb, _stream(stream)), "fs_prune_cells")
    return pool, count


def fs_prune_cells_static(amax, N, params=None, pool=None, count=None, stream=None):
    """fs_prune_cells on the library's fixed scratch array (no workspace).
    ``pool`` / ``count`` may be given to avoid allocating outputs here."""
    L = load()
    p = _params(params)
    _dev(amax, "amax", (torch.float32,))
    B, H, C = amax.shape
    nblk = N // p.Bq
    if pool is None:
        pool = torch.empty((B, H, nblk, p.P + p.W), device=amax.device, dtype=torch.int32)
    if count is None:
        count = torch.empty((B, H, nblk), device=amax.device, dtype=torch.int32)
    _check(L.fs_prune_cells_static(_ptr(amax), B, H, N, ctypes.byref(p), _ptr(pool),
                                   _ptr(count), _stream(stream)), "fs_prune_cells_static")
    return pool, count


def fs_selftest_wait_timeout(ws, stream=None):
    """Launch the bounded-wait self-test into workspace ``ws`` (device uint8,
    >= 256 bytes); read the outcome with fs_check_status(ws)."""
    _check(load().fs_selftest_wait_timeout(_ptr(ws), _stream(stream)), "fs_selftest_wait_timeout")


def fs_decode_state_bytes(batch, H, d=64, params=None) -> int:
    p = _params(params)
    return load().fs_decode_state_bytes(batch, H, d, ctypes.byref(p))


def fs_decode_state_view(state, batch, H, params=None):
    """Views into a decode state: per (batch, head) slot cell ids [BH, nslots]
    int32, slot a_c [BH, nslots] f32, slot mean keys [BH, nslots, 64] f32,
    and the header ints [BH, n] (position, list counts, lists)."""
    L = load()
    p = _params(params)
    offs = (ctypes.c_size_t * 7)()
    _check(L.fs_decode_state_view(batch, H, 64, ctypes.byref(p), offs), "fs_decode_state_view")
    g, hb, oc, oa, ok, ns, nh = (int(x) for x in offs)
    heads = state[g:g + batch * H * hb].view(batch * H, hb)
    return dict(cell=heads[:, oc:oc + 4 * ns].contiguous().view(torch.int32),
                amax=heads[:, oa:oa + 4 * ns].contiguous().view(torch.float32),
                kbar=heads[:, ok:ok + 4 * 64 * ns].contiguous().view(torch.float32).view(-1, ns, 64),
                header=heads[:, :4 * nh].contiguous().view(torch.int32))


def fs_decode_state_init(batch, H, params=None, k=None, v=None, kbar=None, amax=None, pool=None,
                         pool_count=None, N0=0, state=None, device=None, stream=None):
    """Bounded decode state after the first N0 tokens (N0 = 0: an empty state).
    For N0 > 0, k, v [B,H,N,d] bf16 hold the prefix in rows < N0, and kbar,
    amax, pool, pool_count are fs_cell_summarize / fs_prune_cells of k.
    Returns the state (a device uint8 tensor of fs_decode_state_bytes)."""
    L = load()
    p = _params(params)
    nb = L.fs_decode_state_bytes(batch, H, 64, ctypes.byref(p))
    if nb == 0:
        raise FSError(FS_ERR_INVALID_ARG, "fs_decode_state_bytes")
    if N0 > 0:
        for t_, n in ((k, "k"), (v, "v")):
            _dev(t_, n, (torch.bfloat16,))
        for t_, n in ((kbar, "kbar"), (amax, "amax")):
            _dev(t_, n, (torch.float32,))
        for t_, n in ((pool, "pool"), (pool_count, "pool_count")):
            _dev(t_, n, (torch.int32,))
        N = k.shape[2]
        device = k.device
    else:
        N = 128
        device = device or torch.device("cuda")
    if state is None:
        state = torch.empty(nb, device=device, dtype=torch.uint8)
    elif state.numel() * state.element_size() < nb:
        raise ValueError(f"state too small: {state.numel()} < {nb} bytes")
    _check(L.fs_decode_state_init(_ptr(k), _ptr(v), FS_BF16, _ptr(kbar), _ptr(amax), _ptr(pool),
                                  _ptr(pool_count), batch, H, N, int(N0), 64, ctypes.byref(p),
                                  _ptr(state), nb, _stream(stream)), "fs_decode_state_init")
    return state


def fs_decode_step(q_t, k_t, v_t, t, state, lam, sigma, mix, params=None, out=None,
                   sel=None, stream=None):
    """One decode step for token t from the bounded ``state`` (advanced in
    place).  q_t, k_t, v_t [B,H,d] bf16.  Returns out_t [B,H,d] f32."""
    L = load()
    p = _params(params)
    for t_, n in ((q_t, "q_t"), (k_t, "k_t"), (v_t, "v_t")):
        _dev(t_, n, (torch.bfloat16,))
    B, H, d = q_t.shape
    out = out if out is not None else torch.empty((B, H, d), device=q_t.device, dtype=torch.float32)
    _check(L.fs_decode_step(_ptr(q_t), _ptr(k_t), _ptr(v_t), FS_BF16, B, H, d, int(t), _ptr(lam),
                            _ptr(sigma), _ptr(mix), ctypes.byref(p), _ptr(state),
                            state.numel() * state.element_size(), _ptr(out), _ptr(sel),
                            _stream(stream)), "fs_decode_step")
    return out


def fs_fsb_select(q, k, kbar, amax, lam, sigma, params=None, stream=None):
    """FS-B selection (beam search over the two forests, token rerank):
    sel [B,H,N,K] int32.  params.mode must be FS_MODE_FSB."""
    L = load()
    p = _params(params)
    for t_, n in ((q, "q"), (k, "k")):
        _dev(t_, n, (torch.bfloat16,))
    for t_, n in ((kbar, "kbar"), (amax, "amax"), (lam, "lam"), (sigma, "sigma")):
        _dev(t_, n, (torch.float32,))
    B, H, N, d = _qkv_shape(q)
    wsb = L.fs_fsb_workspace_bytes(B, H, N, ctypes.byref(p))
    if wsb == 0:
        raise FSError(FS_ERR_INVALID_ARG, "fs_fsb_workspace_bytes")
    ws = torch.empty(wsb, device=q.device, dtype=torch.uint8)
    sel = torch.empty((B, H, N, p.K), device=q.device, dtype=torch.int32)
    _check(L.fs_fsb_select(_ptr(q), _ptr(k), _ptr(kbar), _ptr(amax), _ptr(lam), _ptr(sigma), B, H,
                           N, d, ctypes.byref(p), _ptr(sel), _ptr(ws), wsb, _stream(stream)),
           "fs_fsb_select")
    return sel


def fs_backward_workspace_bytes(batch, H, N, d=64, params=None) -> int:
    p = _params(params)
    return load().fs_backward_workspace_bytes(batch, H, N, d, ctypes.byref(p))


def fs_attention_bwd(q, k, v, lam, sigma, mix, dout, params=None, ws=None, stream=None):
    """Gradients of L = sum(dout * fs_attention_fwd(q, k, v, ...)) with the
    forward's selections held fixed.  Returns dq, dk, dv [B,H,N,d] f32 and
    dmix [H] f32."""
    L = load()
    p = _params(params)
    for t_, n in ((q, "q"), (k, "k"), (v, "v")):
        _dev(t_, n, (torch.bfloat16,))
    _dev(dout, "dout", (torch.float32,))
    for t_, n in ((lam, "lam"), (sigma, "sigma"), (mix, "mix")):
        _dev(t_, n, (torch.float32,))
    B, H, N, d = _qkv_shape(q)
    wsb = L.fs_backward_workspace_bytes(B, H, N, d, ctypes.byref(p))
    if wsb == 0:
        raise FSError(FS_ERR_INVALID_ARG, "fs_backward_workspace_bytes")
    if ws is None:
        ws = torch.empty(wsb, device=q.device, dtype=torch.uint8)
    dq, dk, dv = (torch.empty((B, H, N, d), device=q.device, dtype=torch.float32) for _ in range(3))
    dmix = torch.empty(H, device=q.device, dtype=torch.float32)
    _check(L.fs_attention_bwd(_ptr(q), _ptr(k), _ptr(v), FS_BF16, B, H, N, d, ctypes.byref(p),
                              _ptr(lam), _ptr(sigma), _ptr(mix), _ptr(dout), _ptr(dq), _ptr(dk),
                              _ptr(dv), _ptr(dmix), _ptr(ws), wsb, _stream(stream)),
           "fs_attention_bwd")
    return dq, dk, dv, dmix


def fs_qkv_workspace_bytes(batch, N, D, H) -> int:
    return load().fs_qkv_workspace_bytes(batch, N, D, H)


def fs_qkv_prologue(x, w_qkv, H, gain=None, eps=1e-6, q=None, k=None, v=None, ws=None,
                    stream=None):
    """RMSNorm(x) . w_qkv^T split into q, k, v [batch, H, N, 64] bf16.
    x [batch, N, D] bf16, w_qkv [3*H*64, D] bf16, gain [D] f32 or None."""
    L = load()
    _dev(x, "x", (torch.bfloat16,))
    _dev(w_qkv, "w_qkv", (torch.bfloat16,))
    if gain is not None:
        _dev(gain, "gain", (torch.float32,))
    B, N, D = x.shape
    if tuple(w_qkv.shape) != (3 * H * 64, D):
        raise ValueError(f"w_qkv must be [{3 * H * 64}, {D}]")
    outs = []
    for t_ in (q, k, v):
        t_ = t_ if t_ is not None else torch.empty((B, H, N, 64), device=x.device,
                                                   dtype=torch.bfloat16)
        _dev(t_, "q/k/v", (torch.bfloat16,))
        outs.append(t_)
    wsb = L.fs_qkv_workspace_bytes(B, N, D, H)
    if wsb == 0:
        raise FSError(FS_ERR_INVALID_ARG, "fs_qkv_workspace_bytes")
    if ws is None:
        ws = torch.empty(wsb, device=x.device, dtype=torch.uint8)
    _check(L.fs_qkv_prologue(_ptr(x), _ptr(gain), _ptr(w_qkv), B, N, D, H, float(eps),
                             _ptr(outs[0]), _ptr(outs[1]), _ptr(outs[2]), _ptr(ws), wsb,
                             _stream(stream)), "fs_qkv_prologue")
    return tuple(outs)


def fs_select_cells(q, kbar, amax, pool, pool_count, lam, sigma, params=None,
                    with_scores=False, stream=None):
    L = load()
    p = _params(params)
    _dev(q, "q", (torch.bfloat16,))
    B, H, N, d = _qkv_shape(q)
    for t, n in ((kbar, "kbar"), (amax, "amax"), (lam, "lam"), (sigma, "sigma")):
        _dev(t, n, (torch.float32,))
    if pool is not None:
        _dev(pool, "pool", (torch.int32,))
        _dev(pool_count, "pool_count", (torch.int32,))
    sel = torch.empty((B, H, N, p.K), device=q.device, dtype=torch.int32)
    score = torch.empty((B, H, N, p.K), device=q.device, dtype=torch.float32) if with_scores else None
    _check(L.fs_select_cells(_ptr(q), FS_BF16, _ptr(kbar), _ptr(amax), _ptr(pool),
                             _ptr(pool_count), _ptr(lam), _ptr(sigma), B, H, N, d,
                             ctypes.byref(p), _ptr(sel), _ptr(score), _stream(stream)),
           "fs_select_cells")
    return (sel, score) if with_scores else sel


def fs_sparse_readout(q, k, v, sel, params=None, o_long=None, stream=None):
    L = load()
    p = _params(params)
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _dev(t, n, (torch.bfloat16,))
    _dev(sel, "sel", (torch.int32,))
    B, H, N, d = _qkv_shape(q)
    o_long = o_long if o_long is not None else torch.empty((B, H, N, d), device=q.device, dtype=torch.float32)
    _check(L.fs_sparse_readout(_ptr(q), _ptr(k), _ptr(v), FS_BF16, _ptr(sel), B, H, N, d,
                               ctypes.byref(p), _ptr(o_long), _stream(stream)), "fs_sparse_readout")
    return o_long


def fs_window_attn(q, k, v, o_long=None, mix=None, params=None, out=None, stream=None,
                   ws=None, events=None):
    """Window branch (and mix with ``o_long`` when given).  ``events``: None,
    or 3 torch.cuda.Event objects (enable_timing) recorded before the operand
    preparation, before the attention kernel and after it."""
    L = load()
    p = _params(params)
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _dev(t, n, (torch.bfloat16,))
    B, H, N, d = _qkv_shape(q)
    if o_long is not None:
        _dev(o_long, "o_long", (torch.float32,))
        _dev(mix, "mix", (torch.float32,))
    out = out if out is not None else torch.empty((B, H, N, d), device=q.device, dtype=torch.float32)
    wsb = L.fs_window_workspace_bytes(B, H, N, d, ctypes.byref(p))
    if wsb == 0:
        raise FSError(FS_ERR_INVALID_ARG, "fs_window_workspace_bytes")
    if ws is None:
        ws = torch.empty(wsb, device=q.device, dtype=torch.uint8)
    elif ws.numel() * ws.element_size() < wsb:
        raise ValueError(f"workspace too small: {ws.numel()} < {wsb} bytes")
    args = [_ptr(q), _ptr(k), _ptr(v), FS_BF16, _ptr(o_long), _ptr(mix), B, H, N, d,
            ctypes.byref(p), _ptr(out), _ptr(ws), wsb, _stream(stream)]
    if events is None:
        _check(L.fs_window_attn(*args), "fs_window_attn")
    else:
        if len(events) != 3:
            raise ValueError("need 3 events")
        _check(L.fs_window_attn_traced(*args, _event_array(events)), "fs_window_attn_traced")
    return out


def _event_array(events):
    for e in events:
        if e.cuda_event == 0:  # torch creates the CUDA event lazily
            e.record()
    return (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])


def fs_attention_fwd(q, k, v, lam, sigma, mix, params=None, out=None, ws=None, stream=None):
    """Whole FS-L (or FS) forward.  Returns ``out`` [batch, H, N, d] fp32."""
    L = load()
    p = _params(params)
    dt = (torch.bfloat16, torch.float32)
    _dev(q, "q", dt)
    _dev(k, "k", (q.dtype,))
    _dev(v, "v", (q.dtype,))
    for t, n in ((lam, "lam"), (sigma, "sigma"), (mix, "mix")):
        _dev(t, n, (torch.float32,))
    B, H, N, d = _qkv_shape(q)
    code = _dtype_code(q)
    wsb = L.fs_workspace_bytes(B, H, N, d, ctypes.byref(p), code)
    if wsb == 0:
        raise FSError(FS_ERR_INVALID_ARG, "fs_workspace_bytes")
    if ws is None:
        ws = torch.empty(wsb, device=q.device, dtype=torch.uint8)
    elif ws.numel() * ws.element_size() < wsb:
        raise ValueError(f"workspace too small: {ws.numel()} < {wsb} bytes")
    out = out if out is not None else torch.empty((B, H, N, d), device=q.device, dtype=torch.float32)
    _dev(out, "out", (torch.float32,))
    _check(L.fs_attention_fwd(_ptr(q), _ptr(k), _ptr(v), code, B, H, N, d, ctypes.byref(p),
                              _ptr(lam), _ptr(sigma), _ptr(mix), _ptr(out), _ptr(ws), wsb,
                              _stream(stream)), "fs_attention_fwd")
    return out


def fs_host_workspace_bytes(batch, H, N, d, params=None, dtype=FS_BF16, heads_per_chunk=2) -> int:
    p = _params(params)
    return load().fs_host_workspace_bytes(batch, H, N, d, ctypes.byref(p), dtype, heads_per_chunk)


def _host(t, name, dtypes):
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} must have dtype in {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def fs_attention_fwd_host(q, k, v, lam, sigma, mix, params=None, out=None, ws=None,
                          heads_per_chunk=2, stream=None):
    """fs_attention_fwd on host tensors q, k, v [batch, H, N, d] (pinned memory
    lets the copies overlap the compute); lam, sigma, mix are device tensors.
    Returns ``out`` [batch, H, N, d] fp32 on the host, readable after the
    stream is synchronised."""
    L = load()
    p = _params(params)
    for t, nm in ((q, "q"), (k, "k"), (v, "v")):
        _host(t, nm, (torch.bfloat16, torch.float32))
    if not (q.dtype == k.dtype == v.dtype) or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must share dtype and shape")
    for t, nm in ((lam, "lam"), (sigma, "sigma"), (mix, "mix")):
        _dev(t, nm, (torch.float32,))
    B, H, N, d = _qkv_shape(q)
    code = FS_FP32 if q.dtype == torch.float32 else FS_BF16
    wsb = L.fs_host_workspace_bytes(B, H, N, d, ctypes.byref(p), code, heads_per_chunk)
    if wsb == 0:
        raise FSError(FS_ERR_INVALID_ARG, "fs_host_workspace_bytes")
    dev = lam.device
    if ws is None:
        ws = torch.empty(wsb, device=dev, dtype=torch.uint8)
    elif ws.numel() * ws.element_size() < wsb:
        raise ValueError(f"workspace too small: {ws.numel()} < {wsb} bytes")
    if out is None:
        out = torch.empty((B, H, N, d), dtype=torch.float32, pin_memory=True)
    _host(out, "out", (torch.float32,))
    _check(L.fs_attention_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), code, B, H, N, d,
                                   ctypes.byref(p), _ptr(lam), _ptr(sigma), _ptr(mix),
                                   out.data_ptr(), heads_per_chunk, _ptr(ws), wsb,
                                   _stream(stream)), "fs_attention_fwd_host")
    return out


def fs_attention_fwd_traced(q, k, v, lam, sigma, mix, events, params=None, out=None, ws=None,
                            stream=None):
    """fs_attention_fwd recording ``events`` (FS_N_STAGES + 1 torch.cuda.Event
    objects, created with enable_timing) between its stages on the stream."""
    L = load()
    p = _params(params)
    if len(events) != FS_N_STAGES + 1:
        raise ValueError(f"need {FS_N_STAGES + 1} events")
    B, H, N, d = _qkv_shape(q)
    code = _dtype_code(q)
    wsb = L.fs_workspace_bytes(B, H, N, d, ctypes.byref(p), code)
    if wsb == 0:
        raise FSError(FS_ERR_INVALID_ARG, "fs_workspace_bytes")
    if ws is None:
        ws = torch.empty(wsb, device=q.device, dtype=torch.uint8)
    elif ws.numel() * ws.element_size() < wsb:
        raise ValueError("workspace too small")
    out = out if out is not None else torch.empty((B, H, N, d), device=q.device, dtype=torch.float32)
    arr = _event_array(events)
    _check(L.fs_attention_fwd_traced(_ptr(q), _ptr(k), _ptr(v), code, B, H, N, d,
                                     ctypes.byref(p), _ptr(lam), _ptr(sigma), _ptr(mix),
                                     _ptr(out), _ptr(ws), wsb, _stream(stream), arr),
           "fs_attention_fwd_traced")
    return out


def fs_workspace_view(ws, batch, H, N, d, params=None, dtype=FS_BF16):
    """Views of the intermediates an fs_attention_fwd call left in ``ws``:
    dict with kbar, amax, pool, pool_count, sel."""
    L = load()
    p = _params(params)
    offs = [ctypes.c_size_t() for _ in range(5)]
    _check(L.fs_workspace_view(batch, H, N, d, ctypes.byref(p), dtype,
                               *[ctypes.byref(o) for o in offs]), "fs_workspace_view")
    C, nblk = N // p.s, N // p.Bq
    spec = [("kbar", (batch, H, C, d), torch.float32), ("amax", (batch, H, C), torch.float32),
            ("pool", (batch, H, nblk, p.P + p.W), torch.int32),
            ("pool_count", (batch, H, nblk), torch.int32),
            ("sel", (batch, H, N, p.K), torch.int32)]
    res = {}
    for (name, shape, dtype_), off in zip(spec, offs):
        n = 1
        for x in shape:
            n *= x
        nbytes = n * torch.tensor([], dtype=dtype_).element_size()
        res[name] = ws[off.value: off.value + nbytes].view(dtype_).view(shape)
    return res


def fs_set_attention_timeline(buf=None):
    """Record each CTA's start and end (device global timer, ns) of the calling
    thread's following attention launches into ``buf`` (a CUDA int64 tensor,
    two entries per CTA); ``None`` turns it off."""
    global _timeline_buf
    L = load()
    if buf is None:
        _check(L.fs_set_attention_timeline(None, 0), "fs_set_attention_timeline")
        _timeline_buf = None
        return
    if not (buf.is_cuda and buf.dtype == torch.int64 and buf.is_contiguous()):
        raise ValueError("timeline must be a contiguous CUDA int64 tensor")
    _check(L.fs_set_attention_timeline(_ptr(buf), buf.numel()), "fs_set_attention_timeline")
    _timeline_buf = buf  # the library keeps only the pointer: keep the memory alive


_timeline_buf = None


def fs_check_status(ws, stream=None):
    """Synchronise the stream and raise FSError if a kernel recorded an error
    (a bounded device wait that timed out) in the workspace header."""
    _check(load().fs_check_status(_ptr(ws), _stream(stream)), "fs_check_status")
