"""Benchmark of the FS-L attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload fsl_64k]
                    [--impl ours|reference] [--no-cpu-baseline] [--no-e2e]

One step = one ``fs_attention_fwd`` over the whole workload (cell summaries,
pruning, selection, readout, window + mix), inputs resident in HBM.  With
``--gpus N`` (under torchrun) every rank runs its own replica of the workload
on its GPU (the op shards over independent (batch, head) slices, so there is
no data-path collective): weak scaling, value = tokens of all ranks / max
rank time.  Prints one JSON line on rank 0.

``--impl reference`` times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload (rank 0 only) and prints the same kind of line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from long_context_lm_gb300.inputs import WORKLOADS, make_inputs  # noqa: E402

METRIC = "FS-L attn fwd tokens/s at 16k/64k/256k (H=16,d=64,bf16); % of roofline"
UNIT = "tokens/s"
L2_BYTES = 129 * 1024 * 1024
STAGE_STEPS = 50  # traced steps for the per-stage times, after the timed region
E2E_HEADS = 2  # heads per group of the host-buffer pipeline (2.60 ms per call vs 2.73 for 4, 3.15 for 8)
# dram__bytes_read.sum + dram__bytes_write.sum of fs_attn_tc_kernel in one ncu
# capture (fsl_16k_b2: 281.92 + 106.35 MB over 2*16*16384 token-heads)
ATTN_DRAM_BYTES_PER_TOKEN_HEAD = (281.918208e6 + 106.351104e6) / (2 * 16 * 16384)


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def combine_ranks(ms, tokens_per_rank, world, device):
    """Whole-job figure of a weak-scaling run: every rank processed
    `tokens_per_rank` in `ms`; the job time is the slowest rank's (max over
    ranks) and the throughput counts the tokens of all ranks."""
    if world > 1:
        t = torch.tensor([ms], device=device, dtype=torch.float64)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    return ms, tokens_per_rank * world / (ms / 1e3)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"],
                    bf16_sustained=d.get("bf16_tflops_sustained"), source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def window_flops(BH, N, w, d=64):
    """Algorithmic flops of the window branch: QK^T and PV over the exact
    number of keys each query attends to (4*d per query-key pair)."""
    n = np.arange(N, dtype=np.float64)
    return float(BH * 4 * d * np.minimum(n + 1, w).sum())


def stage_work(wl, distinct_cells, sel_counts):
    """Algorithmic bytes / flops per launch of each stage (one step)."""
    B, H, N, d = wl.batch, wl.heads, wl.seq_len, wl.head_dim
    BH, C, nblk = B * H, N // 32, N // 128
    p = wl.params
    K, cap = p["K"], p["P"] + p["W"]
    tok = BH * N
    work = {}
    # one pass: read k, v; write the cell summaries (kbar fp32 and amax), the
    # rotated keys as bf16 hi | lo and v as fp16
    work["cells_prep"] = dict(bound="hbm", bytes=tok * d * 2 * 2 + BH * C * (d * 4 + 4)
                              + tok * d * 2 * 3)
    # prune: read amax (chunk sort + per block), write pools
    work["prune"] = dict(bound="latency", bytes=BH * C * 4 * 2 + BH * nblk * (cap + 1) * 4)
    # select: q (bf16), pool ids, mean keys of the pool cells once per block
    # (fp32), sel out; flops: q.kbar for every candidate of every query
    work["select"] = dict(bound="tensor", bytes=tok * d * 2 + BH * nblk * cap * (d * 4 + 8) + tok * K * 4,
                          flops=2.0 * d * float(sel_counts["cands"]))
    # attention (both branches + mix): q (bf16), rotated keys (bf16 hi | lo),
    # fp16 values, sel, out (fp32), the raw k/v of every distinct selected
    # cell once; flops: QK^T and PV over the window keys of every query plus
    # the tokens of its selected cells
    work["attention"] = dict(bound="tensor",
                             bytes=tok * d * (2 + 4 + 2 + 4) + tok * K * 4
                             + distinct_cells * 32 * d * 2 * 2,
                             flops=window_flops(BH, N, p["w"], d) + 4.0 * d * float(sel_counts["tokens_read"]))
    return work


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args, rank, world, local_rank):
    from long_context_lm_gb300 import fs
    from long_context_lm_gb300.fs import FS_N_STAGES, STAGE_NAMES

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = WORKLOADS[args.workload]
    inp = make_inputs(wl.batch, wl.heads, wl.seq_len, wl.head_dim, wl.seed, wl.sigma_ln, wl.dtype,
                      wl.needles, wl.n_needles, wl.params)
    B, H, N, d = inp.q.shape
    params = fs.fs_default_params(**wl.params)
    code = fs.FS_FP32 if inp.q.dtype == torch.float32 else fs.FS_BF16
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    lam, sigma, mix = inp.lam.to(dev), inp.sigma.to(dev), inp.mix.to(dev)
    ws = torch.empty(fs.fs_workspace_bytes(B, H, N, d, params, code), device=dev, dtype=torch.uint8)
    out = torch.empty((B, H, N, d), device=dev, dtype=torch.float32)
    stream = torch.cuda.current_stream(dev)
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v))

    # warm-up (also builds the selection statistics used for the byte counts)
    for _ in range(args.warmup):
        fs.fs_attention_fwd(q, k, v, lam, sigma, mix, params, out=out, ws=ws)
    torch.cuda.synchronize()
    view = fs.fs_workspace_view(ws, B, H, N, d, params, code)
    sel = view["sel"].reshape(B * H, -1)
    distinct = sum(int(torch.unique(sel[i][sel[i] >= 0]).numel()) for i in range(B * H))
    nsel = int((view["sel"] >= 0).sum().item())
    if params.mode == fs.FS_MODE_FSL:
        cands = int(view["pool_count"].sum().item()) * 128
    else:
        A = torch.arange(N // 128, dtype=torch.float64) * 4
        cands = float(A.sum().item()) * 128 * B * H
    counts = dict(cands=cands, tokens_read=nsel * 32)
    work = stage_work(wl, distinct, counts)

    # timed region: K steps of the plain API call (the per-stage events of the
    # traced call would add about 22 us a step to what is timed)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(args.steps):
            fs.fs_attention_fwd(q, k, v, lam, sigma, mix, params, out=out, ws=ws)
        t1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        total_ms = t0.elapsed_time(t1)
    ms, value = combine_ranks(total_ms / args.steps, B * N, world, dev)
    # the stage breakdown: the same step with CUDA events between its stages,
    # after the timed region
    n_traced = min(args.steps, STAGE_STEPS)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(FS_N_STAGES + 1)]
              for _ in range(n_traced)]
    for i in range(n_traced):
        fs.fs_attention_fwd_traced(q, k, v, lam, sigma, mix, events[i], params, out=out, ws=ws)
    torch.cuda.synchronize()
    stage_ms = {name: statistics.mean(ev[j].elapsed_time(ev[j + 1]) for ev in events)
                for j, name in enumerate(STAGE_NAMES)}

    # end to end through the public API with host buffers: fs_attention_fwd_host
    # takes pinned host q, k, v and returns out in pinned host memory, its
    # copies pipelined with the compute over groups of E2E_HEADS heads
    e2e = None
    if not args.no_e2e:
        hq, hk, hv = (t.pin_memory() for t in (inp.q, inp.k, inp.v))
        hout = torch.empty((B, H, N, d), dtype=torch.float32).pin_memory()
        ws_h = torch.empty(fs.fs_host_workspace_bytes(B, H, N, d, params, code, E2E_HEADS),
                           device=dev, dtype=torch.uint8)
        e2e_steps = max(2, min(args.steps, 5))
        fs.fs_attention_fwd_host(hq, hk, hv, lam, sigma, mix, params, out=hout, ws=ws_h,
                                 heads_per_chunk=E2E_HEADS)  # first call: copy streams
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(e2e_steps):
            fs.fs_attention_fwd_host(hq, hk, hv, lam, sigma, mix, params, out=hout, ws=ws_h,
                                     heads_per_chunk=E2E_HEADS)
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms = a.elapsed_time(b) / e2e_steps
        e2e = {"value": B * N * world / (e2e_ms / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": out.numel() * 4,
               "ms_per_step": e2e_ms,
               "path": f"fs_attention_fwd_host, pinned host buffers, groups of {E2E_HEADS} heads"}
        del ws_h

    pk = peaks()
    kernels = {}
    for name in STAGE_NAMES:
        wk = work[name]
        t_s = stage_ms[name] / 1e3
        entry = {"ms": stage_ms[name], "share": stage_ms[name] / sum(stage_ms.values())}
        entry["GB/s"] = wk["bytes"] / t_s / 1e9
        entry["hbm_frac"] = entry["GB/s"] / pk["hbm"]
        if "flops" in wk:
            entry["TFLOP/s"] = wk["flops"] / t_s / 1e12
            entry["tensor_frac"] = entry["TFLOP/s"] / pk["bf16"]
        entry["bound"] = wk["bound"]
        kernels[name] = entry
    dom = max(STAGE_NAMES, key=lambda n: stage_ms[n])
    wk = work[dom]
    if wk["bound"] == "tensor":
        ach = wk["flops"] / (stage_ms[dom] / 1e3) / 1e12
        traffic = None
        if dom == "attention" and params.mode == fs.FS_MODE_FSL:
            # DRAM bytes per launch: the per-token figure of one ncu capture of
            # the attention kernel on fsl_16k_b2, scaled by the tokens one
            # launch processes
            traffic = ATTN_DRAM_BYTES_PER_TOKEN_HEAD * B * H * N
        roof = {"kernel": dom, "bound": "tensor", "achieved": ach, "peak": pk["bf16"],
                "unit": "TFLOP/s", "frac": ach / pk["bf16"], "traffic": traffic,
                "peak_source": pk["source"] + " (bf16 burst)"}
    else:
        ach = wk["bytes"] / (stage_ms[dom] / 1e3) / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": pk["hbm"], "unit": "GB/s",
                "frac": ach / pk["hbm"], "traffic": None, "peak_source": pk["source"]}
    # our kernels per step: RoPE angle table 1, one pass for the window operands
    # and the cell summaries 1, prune (sort + scan in one kernel per head up to
    # 192 chunks of 64 cells, else sort and, for more than one chunk, scan;
    # then emit), select 1, attention 1 (+3 roundings for fp32 inputs)
    nch = (N // 32 + 63) // 64
    prune_launches = 0 if params.mode == fs.FS_MODE_FS else (
        2 if nch <= 192 else 3)
    launches_per_step = 2 + prune_launches + 1 + 1 + (3 if code == fs.FS_FP32 else 0)
    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if code == fs.FS_BF16 else "fp32",
        "data": "synthetic (seeded; lognormal key norms)",
        "config": {"workload": wl.name, "batch": B, "heads": H, "seq_len": N, "head_dim": d,
                   "w": params.w, "s": params.s, "K": params.K, "P": params.P, "W": params.W,
                   "Bq": params.Bq, "mode": ["FS-L", "FS", "FS-B"][params.mode],
                   "parallelism": f"replica x{world} (independent (batch, head) slices)",
                   "l2": "inputs larger than L2 (%.0f MB vs 129 MB)" % (in_bytes / 2**20)},
        "roofline": roof, "kernels": kernels, "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_extras:
        res["branches"] = time_branches(q, k, v, mix, view["sel"], params, stream, distinct,
                                        counts, pk)
    if not args.no_extras or getattr(args, "decode_only", False):
        res["decode"] = time_decode(q, k, v, lam, sigma, mix, params, stream)
    if not args.no_extras:
        res["fs_mode"] = time_fs_mode(q, k, v, lam, sigma, mix, params, stream, B * N)
        res["fsb_mode"] = time_fsb_mode(q, k, v, lam, sigma, mix, params, stream, B * N)
        res["prologue"] = time_prologue(B, N, H, stream)
        res["backward"] = time_backward(q, k, v, lam, sigma, mix, params, stream, counts)
        res["graph"] = time_graph(q, k, v, lam, sigma, mix, params, stream, out, ws,
                                  min(args.steps, 100))
    return res


def time_graph(q, k, v, lam, sigma, mix, params, stream, out, ws, steps):
    """The same forward captured once in a CUDA graph and replayed back to
    back on the benchmark's inputs: one graph launch a step instead of the
    call's six kernel launches (a warm-up call on the capturing stream
    precedes the capture, as the graph test does)."""
    from long_context_lm_gb300 import fs
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        fs.fs_attention_fwd(q, k, v, lam, sigma, mix, params, out=out, ws=ws)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fs.fs_attention_fwd(q, k, v, lam, sigma, mix, params, out=out, ws=ws)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    B, _, N, _ = q.shape
    return {"ms_per_step": ms, "tokens_per_s": B * N / (ms / 1e3), "steps": steps,
            "note": "fs_attention_fwd captured once in a CUDA graph, replayed back to back"}


def _timed(fn, stream, iters):
    """Mean device time (ms) of fn() over `iters` back-to-back calls on `stream`
    after two warm-up calls (CUDA events on the launching stream)."""
    for _ in range(2):
        fn()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(iters):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / iters


def _entry(ms, nbytes, flops, pk, bound):
    e = {"ms": ms, "bound": bound, "GB/s": nbytes / (ms / 1e3) / 1e9}
    e["hbm_frac"] = e["GB/s"] / pk["hbm"]
    if flops is not None:
        e["TFLOP/s"] = flops / (ms / 1e3) / 1e12
        e["tensor_frac"] = e["TFLOP/s"] / pk["bf16"]
    return e


def time_branches(q, k, v, mix, sel, params, stream, distinct_cells, counts, pk, iters=20):
    """Each kernel of the path on its own, on the benchmark's inputs, against its
    own roofline: the cell summary (HBM), the window branch alone (prep pass +
    tensor-core kernel, no long branch), and the NoPE readout of the forward's
    own selection alone (the gathered long branch)."""
    from long_context_lm_gb300 import fs
    B, H, N, d = q.shape
    tok = B * H * N
    C = N // 32
    res = {}
    # cell summary: read k (128 B), write kbar (d fp32) and amax per cell
    kbar = torch.empty((B, H, C, d), device=q.device, dtype=torch.float32)
    amax = torch.empty((B, H, C), device=q.device, dtype=torch.float32)
    ms = _timed(lambda: fs.fs_cell_summarize(k, kbar=kbar, amax=amax), stream, iters)
    res["cell_summary"] = _entry(ms, tok * d * 2 + B * H * C * (d * 4 + 4), None, pk, "hbm")
    res["cell_summary"]["bytes_per_token_head"] = (tok * d * 2 + B * H * C * (d * 4 + 4)) / tok
    # window branch alone (o_long = NULL): events around the prep pass and the kernel
    wsb = fs.fs_window_workspace_bytes(B, H, N, d, params)
    ws = torch.empty(wsb, device=q.device, dtype=torch.uint8)
    out = torch.empty((B, H, N, d), device=q.device, dtype=torch.float32)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(iters + 2)]
    for ev in evs:
        fs.fs_window_attn(q, k, v, None, None, params, out=out, ws=ws, events=ev)
    torch.cuda.synchronize()
    prep_ms = statistics.mean(ev[0].elapsed_time(ev[1]) for ev in evs[2:])
    win_ms = statistics.mean(ev[1].elapsed_time(ev[2]) for ev in evs[2:])
    # prep: angle table + read k, v (bf16), write rotated keys (bf16 hi | lo) and fp16 v
    res["window_prep"] = _entry(prep_ms, tok * d * 2 * 2 + tok * d * 2 * 3, None, pk, "hbm")
    # window kernel: q, rotated keys, fp16 values read once, out written (fp32)
    res["window_attn"] = _entry(win_ms, tok * (d * 2 + d * 4 + d * 2 + d * 4),
                                window_flops(B * H, N, params.w, d), pk, "tensor")
    # long branch alone: q, sel, the raw k/v rows of every distinct selected
    # cell once, o_long written (fp32); flops over the selected tokens
    o_long = torch.empty((B, H, N, d), device=q.device, dtype=torch.float32)
    ms = _timed(lambda: fs.fs_sparse_readout(q, k, v, sel, params, o_long=o_long), stream, iters)
    nbytes = tok * (d * 2 + params.K * 4 + d * 4) + distinct_cells * 32 * d * 2 * 2
    res["sparse_readout"] = _entry(ms, nbytes, 4.0 * d * float(counts["tokens_read"]), pk, "hbm")
    del ws, out, o_long
    return res


def time_fsb_mode(q, k, v, lam, sigma, mix, params, stream, tokens, steps=3):
    """FS-B (beam search over the two forests, token rerank) on the same
    inputs; tau = the median cell norm of the inputs (the pages calibrate it
    once per model as a median cell norm)."""
    from long_context_lm_gb300 import fs
    from long_context_lm_gb300.fs import FS_N_STAGES
    _, amax = fs.fs_cell_summarize(k)
    d = {f: getattr(params, f) for f, _ in params._fields_}
    d["mode"] = fs.FS_MODE_FSB
    d["tau"] = float(amax.median().item())
    B, H, N, hd = q.shape
    ws = torch.empty(fs.fs_workspace_bytes(B, H, N, hd, d, fs.FS_BF16), device=q.device,
                     dtype=torch.uint8)
    out = torch.empty((B, H, N, hd), device=q.device, dtype=torch.float32)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(FS_N_STAGES + 1)]
              for _ in range(steps + 1)]
    for i in range(steps + 1):  # the first is a warm-up
        fs.fs_attention_fwd_traced(q, k, v, lam, sigma, mix, events[i], d, out=out, ws=ws)
    torch.cuda.synchronize()
    ms = statistics.mean(ev[0].elapsed_time(ev[-1]) for ev in events[1:])
    sel_ms = statistics.mean(ev[2].elapsed_time(ev[3]) for ev in events[1:])
    # the search's work at full beams and a full union (the design's maximum
    # per query): per forest level 2 * beam node bounds (a 64-term dot with
    # the node mean, 256 B of mean + 16 B of node data), then the token LSE of
    # 2 * beam cells (32 x 64-term dots, 4 KB of keys each).  Forest sizes are
    # the inputs' own: A cells before the block, and of those the ones above
    # tau.
    am = amax.reshape(B * H, -1).float()
    above = torch.cumsum((am > d["tau"]).to(torch.int64), dim=1).cpu().numpy()
    nb = N // 128
    A = np.arange(nb) * 4
    m1 = np.where(A > 0, above[:, np.maximum(A - 1, 0)], 0)  # [BH, nb]
    lv = lambda m: np.where(m > 1, np.ceil(np.log2(np.maximum(m, 1))), 0.0)
    levels = lv(A)[None, :] + lv(m1)  # per (head, block)
    nodes = 128.0 * float((levels * 2 * d["beam"]).sum())
    union = 128.0 * float(((A[None, :] > 0) * 2 * d["beam"]).sum())
    fma = nodes * 64 + union * 32 * 64
    l2 = nodes * (256 + 16) + union * 32 * 64 * 2
    peak = 152 * 128 * 2 * 2.07e9 / 1e12  # TFLOP/s, fp32 FMA
    ach = 2 * fma / (sel_ms / 1e3) / 1e12
    return {"ms_per_step": ms, "tokens_per_s": tokens / (ms / 1e3), "search_ms": sel_ms,
            "tau": d["tau"], "beam": d["beam"], "steps": steps,
            "search_roofline": {"bound": "alu", "achieved_TFLOP/s": ach, "peak_TFLOP/s": peak,
                                "frac": ach / peak, "l2_GB/s": l2 / (sel_ms / 1e3) / 1e9,
                                "note": "work at full beams and union (an upper bound on the "
                                        "executed work); a warp per query reading node means "
                                        "and candidate keys through L2"}}


def time_prologue(B, N, H, stream, D=1024, iters=10):
    """The shared q / k / v projection of a layer with d_model = D feeding the
    benchmark's attention shape (random-init weights, gain folded): one call
    = row-scale pass + gain fold + tcgen05 GEMM, timed with CUDA events."""
    from long_context_lm_gb300 import fs
    from long_context_lm_gb300.inputs import make_prologue_inputs
    inp = make_prologue_inputs(B, N, D, H, seed=11)
    x, w, g = inp.x.cuda(), inp.w_qkv.cuda(), inp.gain.cuda()
    outs = [torch.empty((B, H, N, 64), device=x.device, dtype=torch.bfloat16) for _ in range(3)]
    ws = torch.empty(fs.fs_qkv_workspace_bytes(B, N, D, H), device=x.device, dtype=torch.uint8)
    ms = _timed(lambda: fs.fs_qkv_prologue(x, w, H, gain=g, q=outs[0], k=outs[1], v=outs[2],
                                           ws=ws), stream, iters)
    flops = 2.0 * B * N * D * 3 * H * 64
    pk = peaks()
    return {"ms": ms, "d_model": D, "TFLOP/s": flops / (ms / 1e3) / 1e12,
            "tensor_frac": flops / (ms / 1e3) / 1e12 / pk["bf16"],
            "note": "RMSNorm row scales + gain fold + GEMM [B*N, D] x [D, 3*H*64] bf16 -> q, k, v"}


def time_backward(q, k, v, lam, sigma, mix, params, stream, counts, iters=3):
    """fs_attention_bwd on the benchmark's inputs with a random upstream
    gradient (the forward's selection recomputed inside the call).  Every
    contraction runs on the tensor cores (bf16 operands split hi | lo where
    fp32 inputs need it), so the roofline is the bf16 tensor peak and the
    work the useful flops of the plain algorithm: 640 per (query, window key)
    pair (S, dP, dv, dq, dk: 2 x 64 each) and 768 per (query, selected token)
    pair of the long branch (the same plus the recomputed o)."""
    from long_context_lm_gb300 import fs
    B, H, N, d = q.shape
    g = torch.randn((B, H, N, d), device=q.device, dtype=torch.float32)
    ws = torch.empty(fs.fs_backward_workspace_bytes(B, H, N, d, params), device=q.device,
                     dtype=torch.uint8)
    ms = _timed(lambda: fs.fs_attention_bwd(q, k, v, lam, sigma, mix, g, params, ws=ws), stream,
                iters)
    n = np.arange(N, dtype=np.float64)
    win_pairs = B * H * float(np.minimum(n + 1, params.w).sum())
    flops = 640.0 * win_pairs + 768.0 * float(counts["tokens_read"])
    pk = peaks()
    ach = flops / (ms / 1e3) / 1e12
    return {"ms": ms, "tokens_per_s": B * N / (ms / 1e3), "bound": "tensor",
            "achieved_TFLOP/s": ach, "peak_TFLOP/s": pk["bf16"], "frac": ach / pk["bf16"],
            "note": "tcgen05 kernels (window: query side and key side; long branch: union "
                    "tiles); useful flops; includes recomputing the forward's selection"}


def time_decode(q, k, v, lam, sigma, mix, params, stream, steps=256, warm=8):
    """Decode steps right after the whole prefix: the bounded state is built
    from the prefill (cell summaries, pools, fs_decode_state_init at N0 = N),
    then tokens t = N, N+1, ... are decoded (the new tokens are rows of the
    prefix's last block).  `steps` consecutive steps (two block starts, where
    the pool advances, and eight cell closes) are captured in a CUDA graph
    and replayed once, so the time is the device's, not the host's launch
    rate; the state has the same size at any t."""
    from long_context_lm_gb300 import fs
    B, H, N, d = q.shape
    kbar, amax = fs.fs_cell_summarize(k)
    pool, count = fs.fs_prune_cells(amax, N, params)
    state = fs.fs_decode_state_init(B, H, params, k=k, v=v, kbar=kbar, amax=amax, pool=pool,
                                    pool_count=count, N0=N)
    rows = [N - 128 + (i % 128) for i in range(warm + steps)]
    toks = [tuple(x[:, :, r].contiguous() for x in (q, k, v)) for r in rows]
    out = torch.empty((B, H, d), device=q.device, dtype=torch.float32)
    for i in range(warm):
        fs.fs_decode_step(*toks[i], N + i, state, lam, sigma, mix, params, out=out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s2 = torch.cuda.Stream()
    with torch.cuda.stream(s2):
        with torch.cuda.graph(g, stream=s2):
            for i in range(warm, warm + steps):
                fs.fs_decode_step(*toks[i], N + i, state, lam, sigma, mix, params, out=out)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    fs.fs_check_status(state)
    us = a.elapsed_time(b) / steps * 1e3
    # one step of one (batch, head) reads the new q, k, v (bf16), the window's
    # keys and values (bf16), the candidates' summaries (mean key fp32 and
    # norm) and the K selected cells' keys and values, and writes the output
    # (fp32) and the new token's ring entry
    cap = params.P + params.W
    step_bytes = (3 * d * 2 + params.w * d * 2 * 2 + cap * (d * 4 + 4)
                  + params.K * 32 * d * 2 * 2 + d * 4 + d * 2 * 2)
    pk = peaks()
    gbs = B * H * step_bytes / (us / 1e6) / 1e9
    roof = {"bound": "hbm", "bytes_per_head_step": step_bytes, "GB/s": gbs,
            "hbm_frac": gbs / pk["hbm"],
            "note": "a cluster of 8 CTAs per (batch, head): latency-bound, not "
                    "bandwidth-bound; bytes counted in bf16 (the ring keeps fp32 rotated keys)"}
    return {"t0": N + warm, "us_per_token": us, "heads": B * H, "steps": steps, "roofline": roof,
            "state_bytes": state.numel(), "state_bytes_per_head": state.numel() / (B * H),
            "note": "bounded state from the prefill; graph of consecutive steps, all (batch, head)"}


def time_fs_mode(q, k, v, lam, sigma, mix, params, stream, tokens, steps=3):
    """Base FS (every available cell is a candidate, no pruning) on the same
    inputs: the quadratic comparator of FS-L."""
    from long_context_lm_gb300 import fs
    from long_context_lm_gb300.fs import FS_N_STAGES
    d = {f: getattr(params, f) for f, _ in params._fields_}  # a copy: params stays FS-L
    d["mode"] = fs.FS_MODE_FS
    B, H, N, hd = q.shape
    ws = torch.empty(fs.fs_workspace_bytes(B, H, N, hd, d, fs.FS_BF16), device=q.device,
                     dtype=torch.uint8)
    out = torch.empty((B, H, N, hd), device=q.device, dtype=torch.float32)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(FS_N_STAGES + 1)]
              for _ in range(steps + 1)]
    for i in range(steps + 1):  # the first is a warm-up
        fs.fs_attention_fwd_traced(q, k, v, lam, sigma, mix, events[i], d, out=out, ws=ws)
    torch.cuda.synchronize()
    ms = statistics.mean(ev[0].elapsed_time(ev[-1]) for ev in events[1:])
    sel_ms = statistics.mean(ev[2].elapsed_time(ev[3]) for ev in events[1:])
    # select with every available cell a candidate: each query scores the
    # A = 4 * block cells before its block (flops: q . kbar per candidate);
    # bytes: q, every head's mean keys once, sel out
    nb = N // 128
    cands = B * H * 128.0 * float((np.arange(nb) * 4).sum())
    pk = peaks()
    sel = _entry(sel_ms, B * H * N * hd * 2 + B * H * (N // 32) * (hd * 4 + 4) + B * H * N * d["K"] * 4,
                 2.0 * hd * cands, pk, "tensor")
    sel["candidates"] = cands
    return {"ms_per_step": ms, "tokens_per_s": tokens / (ms / 1e3), "select_ms": sel_ms,
            "select": sel, "steps": steps}


# ---------------------------------------------------------------------------
# oracle on host cores (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------

def oracle_sample(wl, budget_s=10.0, start=0, inp=None):
    """Time the fp64 oracle, as it stands, on the host cores on a bounded
    sample of the workload: whole (batch, head) slices, every query row, one
    slice after another until the time budget is spent (at least one slice).
    Returns (tokens_per_s, cores, description, seconds)."""
    from oracle import oracle as O
    from long_context_lm_gb300.inputs import bf16_values

    O.build()
    if inp is None:
        inp = make_inputs(wl.batch, wl.heads, wl.seq_len, wl.head_dim, wl.seed, wl.sigma_ln,
                          wl.dtype, wl.needles, wl.n_needles, wl.params)
    B, H, N, d = inp.q.shape
    qs, ks, vs = [t.reshape(B * H, N, d) for t in (inp.q, inp.k, inp.v)]
    cores = O.max_threads()
    elapsed, slices = 0.0, 0
    for i in range(B * H):
        bh = (start + i) % (B * H)
        q, k, v = [bf16_values(t[bh:bh + 1]).numpy() for t in (qs, ks, vs)]
        h = bh % H
        t = time.perf_counter()
        O.forward(q, k, v, 1, inp.lam.numpy()[h:h + 1], inp.sigma.numpy()[h:h + 1],
                  inp.mix.numpy()[h:h + 1], params=wl.params, want_branches=False)
        elapsed += time.perf_counter() - t
        slices += 1
        if elapsed >= budget_s:
            break
    # one token = one position of one batch row across all H heads
    tok_per_s = slices * N / H / elapsed
    desc = (f"{slices} of {B * H} (batch, head) slices of {wl.name} (N={N}), every query row; "
            f"tokens counted as rows / H")
    return tok_per_s, cores, desc, elapsed


def run_reference(args):
    wl = WORKLOADS[args.workload]
    inp = make_inputs(wl.batch, wl.heads, wl.seq_len, wl.head_dim, wl.seed, wl.sigma_ln, wl.dtype,
                      wl.needles, wl.n_needles, wl.params)
    per_step = []
    budget = min(10.0, 120.0 / max(1, args.steps + args.warmup))
    cores = desc = None
    for i in range(args.warmup + args.steps):
        v, cores, desc, el = oracle_sample(wl, budget_s=budget, start=i, inp=inp)
        if i >= args.warmup:
            per_step.append(v)
    value = statistics.mean(per_step)
    ms = wl.batch * wl.seq_len / value * 1e3
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 0, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded; lognormal key norms)",
        "impl": "reference",
        "config": {"workload": wl.name, "batch": wl.batch, "heads": wl.heads, "seq_len": wl.seq_len,
                   "head_dim": wl.head_dim, "parallelism": "host cores (OpenMP)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------------------

def probe_calls():
    """One call of each entry point family on small shapes (the fsl_16k_b2
    workload, also each attention branch alone; the projection at B=1, N=16384, D=1024, H=16; four decode steps
    from a state built at N0 = N - 64; FS-B with tau = the median cell norm),
    for profiler captures of every kernel.  Prints nothing but 'ok'."""
    from long_context_lm_gb300 import fs
    from long_context_lm_gb300.inputs import make_prologue_inputs
    wl = WORKLOADS["fsl_16k_b2"]
    inp = make_inputs(wl.batch, wl.heads, wl.seq_len, wl.head_dim, wl.seed, wl.sigma_ln, wl.dtype,
                      wl.needles, wl.n_needles, wl.params)
    d = {k: getattr(inp, k).cuda() for k in ("q", "k", "v", "lam", "sigma", "mix")}
    params = fs.fs_default_params(**wl.params)
    B, H, N, _ = inp.q.shape
    ws = torch.empty(fs.fs_workspace_bytes(B, H, N, 64, params), device="cuda", dtype=torch.uint8)
    fs.fs_attention_fwd(d["q"], d["k"], d["v"], d["lam"], d["sigma"], d["mix"], params, ws=ws)
    # each attention branch alone: the window branch (its operand pass and
    # kernel), and the long branch on the forward's own selection
    sel = fs.fs_workspace_view(ws, B, H, N, 64, params)["sel"].clone()
    fs.fs_window_attn(d["q"], d["k"], d["v"], params=params)
    fs.fs_sparse_readout(d["q"], d["k"], d["v"], sel, params)
    pi = make_prologue_inputs(1, 16384, 1024, 16, seed=1)
    fs.fs_qkv_prologue(pi.x.cuda(), pi.w_qkv.cuda(), 16, gain=pi.gain.cuda())
    kbar, amax = fs.fs_cell_summarize(d["k"])
    pool, cnt = fs.fs_prune_cells(amax, N, params)
    st = fs.fs_decode_state_init(B, H, params, k=d["k"], v=d["v"], kbar=kbar, amax=amax, pool=pool,
                                 pool_count=cnt, N0=N - 64)
    for t in range(N - 64, N - 60):
        fs.fs_decode_step(*(d[x][:, :, t].contiguous() for x in ("q", "k", "v")), t, st, d["lam"],
                          d["sigma"], d["mix"], params)
    g = torch.randn(inp.q.shape, device="cuda")
    fs.fs_attention_bwd(d["q"], d["k"], d["v"], d["lam"], d["sigma"], d["mix"], g, params)
    pb = fs.fs_default_params(**dict(wl.params, mode=fs.FS_MODE_FSB, tau=float(amax.median().item())))
    fs.fs_fsb_select(d["q"], d["k"], kbar, amax, d["lam"], d["sigma"], pb)
    torch.cuda.synchronize()
    fs.fs_check_status(st)
    print("ok")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="fsl_64k", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the decode-step and base-FS timings")
    ap.add_argument("--extra-lengths", default="fsl_16k_b2,fsl_256k",
                    help="other workloads timed briefly for the per-length figures ('none' = skip)")
    ap.add_argument("--probe-calls", action="store_true",
                    help="one call of each entry point on small shapes (for profiler captures), no timing")
    args = ap.parse_args()
    if args.probe_calls:
        probe_calls()
        return
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)))
        return

    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_ours(args, rank, world, local_rank)
    if args.extra_lengths and args.extra_lengths != "none":
        per_len = {args.workload: res["value"]}
        for name in [n for n in args.extra_lengths.split(",") if n and n != args.workload]:
            sub = argparse.Namespace(**vars(args))
            sub.workload, sub.steps, sub.warmup, sub.no_e2e = name, 5, 3, True
            sub.no_extras, sub.decode_only = True, name == "fsl_256k"
            r = run_ours(sub, rank, world, local_rank)
            per_len[name] = r["value"]
            if "decode" in r:
                res["decode_256k"] = r["decode"]
            res.setdefault("other_lengths", {})[name] = {
                "value": r["value"], "ms_per_step": r["ms_per_step"], "roofline": r["roofline"],
                "kernels": {k_: {"ms": v_["ms"], "share": v_["share"]} for k_, v_ in r["kernels"].items()}}
        res["tokens_per_s_by_length"] = per_len
    if rank == 0 and not args.no_cpu_baseline:
        wl = WORKLOADS[args.workload]
        v, cores, desc, el = oracle_sample(wl, budget_s=10.0)
        res["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                               "sample": desc, "seconds": el}
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(res))


if __name__ == "__main__":
    main()
