"""Seeded synthetic workloads for MoE token routing.

This module only draws inputs; it computes nothing the routing method
computes (no selection, no counting, no packing, no combining).  Both the GPU
path and the CPU oracle take their inputs from here, so the two see identical
bytes.

Shapes follow the workloads the pages measure: DeepSeek-V3 and Kimi-K2 style
decode (hidden 7168, 256 / 384 experts, 8 experts per token) and a
Qwen3-235B style prefill (128 experts, 8 per token, hidden 4096) -- see
"Lower latency and higher throughput with multi-node DeepSeek deployment",
section "Expert Parallelism", "Enabling trillion-parameter models on AWS
EFA", section "Evaluation", and "Hosting Qwen on Blackwell", section
"Prefillers".  No dataset is involved: logits and activations are N(0, 1).

Draw order for one workload, from a single CPU ``torch.Generator`` seeded
with ``seed``: logits, then bias (if drawn), then x.
"""
from __future__ import annotations

import dataclasses
import math

import torch

# dtype codes shared with the C ABI (include/moe_route.h)
BF16 = 0
F32 = 1
FP8E4M3_BLK128 = 2

SOFTMAX = 0
SIGMOID = 1

# expert op used by the harness between pack and combine (stands in for the
# grouped expert GEMM, which needs trained weights and is not on this path)
EXPERT_IDENTITY = "identity"
EXPERT_SCALE = "scale"
EXPERT_DEQUANT = "dequant"

# Skewed workload: bias_e = -beta * s * ln(e + 1) with Zipf exponent s = 1.2.
# beta was calibrated once (seed 0) so that the 5% most popular experts draw
# about half of all (token, expert) pairs; a CPU test re-checks the share.
ZIPF_S = 1.2
ZIPF_BETA = 0.535


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    N: int          # virtual ranks (partitions of one GPU's HBM)
    T: int          # tokens per rank
    E: int          # experts
    R: int          # experts per token
    H: int          # hidden size
    x_dtype: int = BF16
    y_dtype: int = BF16
    score_fn: int = SOFTMAX
    renormalize: bool = False
    bias: str = "none"          # "none" | "normal" | "zipf"
    bias_std: float = 0.5
    expert_op: str = EXPERT_IDENTITY
    cap_rows: int = 0           # 0 => default bound N*T*max(R, E/N)
    seed: int = 0

    @property
    def NT(self) -> int:
        return self.N * self.T

    @property
    def L(self) -> int:
        return self.E // self.N

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", N=4, T=64, E=16, R=2, H=1024,
                     score_fn=SOFTMAX, renormalize=False),
    "dsv3_decode": Workload("dsv3_decode", N=32, T=128, E=256, R=8, H=7168,
                            score_fn=SIGMOID, renormalize=True, bias="normal",
                            expert_op=EXPERT_SCALE),
    "qwen3_235b_prefill": Workload("qwen3_235b_prefill", N=4, T=4096, E=128,
                                   R=8, H=4096, score_fn=SOFTMAX,
                                   renormalize=True),
    "kimi_k2_decode": Workload("kimi_k2_decode", N=64, T=64, E=384, R=8,
                               H=7168, score_fn=SOFTMAX, renormalize=True,
                               expert_op=EXPERT_SCALE),
    "skewed": Workload("skewed", N=16, T=1024, E=256, R=8, H=7168,
                       x_dtype=FP8E4M3_BLK128, score_fn=SOFTMAX,
                       renormalize=False, bias="zipf",
                       expert_op=EXPERT_DEQUANT),
}


@dataclasses.dataclass
class Inputs:
    logits: torch.Tensor            # f32 [NT, E]
    bias: torch.Tensor | None       # f32 [E]
    x: torch.Tensor                 # bf16/f32 [NT, H], or uint8 [NT, H] (fp8 codes)
    x_scales: torch.Tensor | None   # f32 [NT, H/128] for fp8


def zipf_bias(E: int, s: float = ZIPF_S, beta: float = ZIPF_BETA) -> torch.Tensor:
    """Deterministic log-Zipf bias, hottest experts at the lowest indices."""
    e = torch.arange(E, dtype=torch.float64)
    return (-beta * s * torch.log(e + 1.0)).to(torch.float32)


def make_inputs(w: Workload, device: str | torch.device = "cpu",
                tie_every: int = 0) -> Inputs:
    """Draw the seeded inputs of workload ``w`` on the CPU (then move them).

    ``tie_every`` > 0 copies, in every ``tie_every``-th token, the logit of
    expert 0 onto expert 1 and expert E-1, so that exact ties in the router
    key occur on purpose (used by the tie-break tests).
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    NT, E, H = w.NT, w.E, w.H
    logits = torch.randn(NT, E, generator=g, dtype=torch.float32)
    if tie_every > 0 and E >= 2 and NT > 0:
        rows = torch.arange(0, NT, tie_every)
        logits[rows, 1] = logits[rows, 0]
        logits[rows, E - 1] = logits[rows, 0]
    bias = None
    if w.bias == "normal":
        bias = torch.randn(E, generator=g, dtype=torch.float32) * w.bias_std
    elif w.bias == "zipf":
        bias = zipf_bias(E)
    x_scales = None
    if w.x_dtype == BF16:
        x = torch.randn(NT, H, generator=g, dtype=torch.float32).to(torch.bfloat16)
    elif w.x_dtype == F32:
        x = torch.randn(NT, H, generator=g, dtype=torch.float32)
    elif w.x_dtype == FP8E4M3_BLK128:
        # activations drawn N(0,1) and stored block-scaled: one fp32 scale per
        # 128 elements (amax / 448, the e4m3 maximum), codes rounded by
        # torch's float8_e4m3fn conversion.
        assert H % 128 == 0
        xf = torch.randn(NT, H // 128, 128, generator=g, dtype=torch.float32)
        amax = xf.abs().amax(dim=2, keepdim=True).clamp_min(1e-12)
        scale = amax / 448.0
        q = (xf / scale).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
        x = q.view(torch.uint8).reshape(NT, H).contiguous()
        x_scales = scale.reshape(NT, H // 128).contiguous()
    else:
        raise ValueError(f"unknown x_dtype {w.x_dtype}")
    inp = Inputs(logits=logits, bias=bias, x=x, x_scales=x_scales)
    if str(device) != "cpu":
        inp = Inputs(*(t.to(device) if t is not None else None
                       for t in (inp.logits, inp.bias, inp.x, inp.x_scales)))
    return inp


def default_cap(w: Workload) -> int:
    """Per-rank receive capacity: the pages' worst case N*T*max(R, E/N)."""
    return w.cap_rows if w.cap_rows > 0 else w.N * w.T * max(w.R, w.E // w.N)


def expert_scale_value(e: int) -> float:
    """Scalar of the 'scale' expert op: 1 + ((e mod 7) - 3)/16 (exact in bf16)."""
    return 1.0 + ((e % 7) - 3) / 16.0


def row_bytes(w: Workload) -> int:
    return {BF16: 2, F32: 4, FP8E4M3_BLK128: 1}[w.x_dtype] * w.H


def y_row_bytes(w: Workload) -> int:
    return {BF16: 2, F32: 4}[w.y_dtype] * w.H


def algorithmic_bytes(w: Workload) -> dict:
    """Bytes each step must move at least once (per launch, whole batch)."""
    NT, R, E, H = w.NT, w.R, w.E, w.H
    rb = row_bytes(w)
    scales_b = 4 * (H // 128) if w.x_dtype == FP8E4M3_BLK128 else 0
    yb = y_row_bytes(w)
    return {
        "route": NT * (4 * E + 8 * R),
        "count": NT * R * 4 * 2,            # read topk_idx, write pos
        "pack": NT * (rb + scales_b) * (1 + R) + NT * R * 8,
        "combine": NT * (yb * R + yb) + NT * R * 8,
    }


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def log_zipf_top_share(counts: torch.Tensor, frac: float = 0.05) -> float:
    """Share of all rows drawn by the top `frac` of experts (by count)."""
    E = counts.numel()
    top = max(1, int(math.floor(frac * E)))
    s = torch.sort(counts.to(torch.float64), descending=True).values
    return float(s[:top].sum() / s.sum())
