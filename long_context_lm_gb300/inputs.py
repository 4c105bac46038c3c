"""Seeded synthetic inputs for the FS-L attention forward.

This module only draws random numbers; it holds none of the method's
arithmetic, so both the CUDA path and the CPU oracle can be fed from it.

Workloads stand in for the long-context retrieval probes the FreeSolo pages
evaluate on (single-needle retrieval, paper.rainbus.top summary, 实验结果):
queries and values are N(0,1); each key is a N(0, I_d) direction scaled per
token by a lognormal(0, sigma_ln) factor, so that cell key norms spread out;
"needle" keys are planted as a multiple of a later query so that the later
query should retrieve them.

Draw order (one CPU ``torch.Generator`` per workload): q, key directions, key
scales, v, lambda, mix, then the needles.  Tensors are drawn in float32 and
rounded once (round-to-nearest-even) to bfloat16 unless the workload is fp32.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

# Method constants of the FS-L variant used by every workload (w, s, K, P, W,
# B) and the RoPE base; sigma_h is the fixed routing sharpness.
FSL_PARAMS = dict(w=512, s=32, K=4, P=64, W=8, Bq=128, rope_base=10000.0,
                  rms_eps=1e-6, mode=0)
SIGMA_H = 4.0


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    heads: int
    seq_len: int
    head_dim: int
    dtype: str            # "fp32" or "bf16": dtype handed to the library
    sigma_ln: float
    needles: str          # "none", "train", "uniform", "deep"
    n_needles: int
    seed: int
    params: dict = field(default_factory=lambda: dict(FSL_PARAMS))


WORKLOADS = {
    # small fp32 case, pure FS in effect (N < (P+W)*s)
    "fsl_2k_h2_fp32": Workload("fsl_2k_h2_fp32", 1, 2, 2048, 64, "fp32", 0.5, "none", 0, 0),
    # training length
    "fsl_4k_b8": Workload("fsl_4k_b8", 8, 16, 4096, 64, "bf16", 0.5, "train", 4, 1),
    # 4x extrapolation, wider key-norm spread
    "fsl_16k_b2": Workload("fsl_16k_b2", 2, 16, 16384, 64, "bf16", 0.8, "uniform", 16, 2),
    # 64k context
    "fsl_64k": Workload("fsl_64k", 1, 16, 65536, 64, "bf16", 0.5, "none", 0, 3),
    # 256k context (64x training length)
    "fsl_256k": Workload("fsl_256k", 1, 16, 262144, 64, "bf16", 0.5, "deep", 1, 4),
}


@dataclass
class Inputs:
    q: torch.Tensor       # [B, H, N, d], bf16 (or fp32 for an fp32 workload)
    k: torch.Tensor
    v: torch.Tensor
    lam: torch.Tensor     # [H] float32
    sigma: torch.Tensor   # [H] float32
    mix: torch.Tensor     # [H] float32
    needles: list         # (b, h, key position p, query position j)
    params: dict


def make_inputs(batch, heads, seq_len, head_dim=64, seed=0, sigma_ln=0.5,
                dtype="bf16", needles="none", n_needles=0, params=None,
                lam_range=(0.5, 1.5), mix_range=(0.0, 1.0)) -> Inputs:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    shape = (batch, heads, seq_len, head_dim)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    xi = torch.randn((batch, heads, seq_len, 1), generator=g, dtype=torch.float32)
    k.mul_(torch.exp(sigma_ln * xi))
    del xi
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    lam = lam_range[0] + (lam_range[1] - lam_range[0]) * torch.rand(heads, generator=g)
    mix = mix_range[0] + (mix_range[1] - mix_range[0]) * torch.rand(heads, generator=g)
    sigma = torch.full((heads,), SIGMA_H, dtype=torch.float32)
    planted = []
    N = seq_len

    def randint(lo, hi):  # uniform integer in [lo, hi)
        return int(torch.randint(lo, hi, (1,), generator=g).item())

    if needles != "none":
        for b in range(batch):
            for h in range(heads):
                for _ in range(n_needles):
                    if needles == "train":      # query j >= 1024, key >= 1024 earlier
                        j = randint(1024, N)
                        p = randint(0, j - 1024 + 1)
                        scale = 3.0
                    elif needles == "uniform":  # key anywhere, query >= 1024 later
                        p = randint(0, N - 1024)
                        j = randint(p + 1024, N)
                        scale = 3.0
                    elif needles == "deep":     # key in [0.05N, 0.5N], last query
                        p = randint(int(0.05 * N), int(0.5 * N) + 1)
                        j = N - 1
                        scale = 12.0            # 3x query, norm boosted 4x
                    else:
                        raise ValueError(needles)
                    k[b, h, p] = scale * q[b, h, j]
                    planted.append((b, h, p, j))
    if dtype == "bf16":
        q, k, v = q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)
    elif dtype != "fp32":
        raise ValueError(dtype)
    return Inputs(q, k, v, lam.float(), sigma, mix.float(), planted,
                  dict(params or FSL_PARAMS))


def workload_inputs(name: str) -> Inputs:
    w = WORKLOADS[name]
    return make_inputs(w.batch, w.heads, w.seq_len, w.head_dim, w.seed, w.sigma_ln,
                       w.dtype, w.needles, w.n_needles, w.params)


def bf16_values(x: torch.Tensor) -> torch.Tensor:
    """The bf16-rounded values of x as float32 (what both sides compute on)."""
    return x.to(torch.bfloat16).to(torch.float32)


@dataclass
class PrologueInputs:
    x: torch.Tensor      # [B, N, D] bf16 hidden states
    gain: torch.Tensor   # [D] float32 RMSNorm gain
    w_qkv: torch.Tensor  # [3*H*d, D] bf16 projection weights (rows: q, k, v heads)


def make_prologue_inputs(batch, seq_len, d_model, heads, head_dim=64, seed=0,
                         gain="random") -> PrologueInputs:
    """Random-init projection inputs: hidden states N(0,1) scaled per token by
    a lognormal(0, 0.5) factor, weights N(0, 1/D) (random initialisation; no
    trained weights exist here), gain U[0.5, 1.5] or ones.  Draw order: x
    directions, token scales, weights, gain."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    x = torch.randn((batch, seq_len, d_model), generator=g, dtype=torch.float32)
    x.mul_(torch.exp(0.5 * torch.randn((batch, seq_len, 1), generator=g, dtype=torch.float32)))
    w = torch.randn((3 * heads * head_dim, d_model), generator=g, dtype=torch.float32)
    w.mul_(d_model ** -0.5)
    if gain == "ones":
        gn = torch.ones(d_model, dtype=torch.float32)
    else:
        gn = 0.5 + torch.rand(d_model, generator=g, dtype=torch.float32)
    return PrologueInputs(x.to(torch.bfloat16), gn, w.to(torch.bfloat16))
