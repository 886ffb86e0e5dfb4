"""Seeded synthetic inputs for the codec's workloads.

This module is shared by the tests, the benchmark and the smoke check, and by
both sides of every parity comparison (the CUDA library and the CPU oracle).
It holds shapes, value distributions and random draws only -- none of the
codec's arithmetic -- and imports neither the oracle nor the library.

The workloads stand in for tensor-parallel activations and gradients of the
kinds the pages describe (TACO: GPT / Qwen TP intermediates; EQuARX: a
standard-normal tensor for its error study; Flash Communication: down-
projection activations with outlier channels).  No dataset is used.

Rank r of a workload draws from a generator seeded with ``seed + r``; the
outlier-channel set is drawn once from ``seed + 1000`` and shared by all ranks.
Values are drawn in float32 on the requested device and rounded once to the
workload's 16-bit dtype by torch's round-to-nearest-even cast.  The bytes
therefore depend on the device the generator ran on; a parity check always
hands the same bytes to both sides.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    ranks: int            # simulated tensor-parallel ranks (separate buffers)
    rows: int             # tokens (or sequence positions)
    cols: int             # hidden size; blocks run along this axis
    dtype: str            # "bf16" or "fp16"
    scheme: str           # reduce-stage scheme
    block: int            # Hadamard block / quantization block or group
    gather_scheme: str    # requantization scheme of the gather stage
    gather_block: int
    dist: str
    params: dict = field(default_factory=dict)
    steps: int = 1        # successive steps (per-step magnitude drift)
    description: str = ""

    @property
    def elems_per_rank(self) -> int:
        return self.rows * self.cols

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float16


WORKLOADS = {
    "taco_tiny": Workload(
        "taco_tiny", 4, 256, 1024, "bf16", "taco_fp8", 128, "taco_fp8", 128,
        "mix_outlier", dict(sigma=0.02, p_out=0.02, sigma_out=1.0, n_chan=8, chan_gain=10.0),
        description="4 TP ranks x [256 x 1024] bf16: 98% N(0,0.02^2) + 2% N(0,1), "
                    "8 fixed hidden channels x10; Hadamard block 128, dual-scale FP8 E4M3"),
    "gpt_tp": Workload(
        "gpt_tp", 8, 8192, 4096, "bf16", "taco_fp8", 128, "taco_fp8", 128,
        "laplace", dict(b=0.01, chan_frac=0.005, chan_gain=20.0),
        description="GPT-style TP row-parallel output: 8 ranks x [2*4096 x 4096] bf16, "
                    "Laplace(0, 0.01), 0.5% of channels x20; Hadamard block 128, FP8 E4M3"),
    "qwen_grad": Workload(
        "qwen_grad", 4, 8192, 5120, "bf16", "taco_fp8", 256, "taco_fp8", 256,
        "normal_drift", dict(sigma=1e-4, lo=0.25, hi=4.0), steps=16,
        description="Qwen-style TP backward gradient: 4 ranks x [8192 x 5120] bf16, "
                    "N(0, 1e-4^2) x per-step log-uniform factor in [0.25, 4], 16 steps; "
                    "Hadamard block 256, FP8 E4M3"),
    "equarx_int8": Workload(
        "equarx_int8", 8, 16384, 8192, "bf16", "int8_sym", 64, "int8_sym", 64,
        "normal", dict(sigma=1.0),
        description="Block-symmetric INT8 reduce-scatter: 8 ranks x [16384 x 8192] bf16 "
                    "N(0,1); one FP32 scale per 64; int8 requantization for the gather"),
    "flash_int4": Workload(
        "flash_int4", 8, 8192, 8192, "fp16", "int4_asym", 128, "int8_asym", 128,
        "student_t", dict(df=3, scale=0.05, chan_frac=0.01, chan_gain=30.0),
        description="Two-stage quantized all-reduce: 8 ranks x [8192 x 8192] fp16 "
                    "down-projection activations, Student-t(3) x 0.05, 1% of channels x30; "
                    "INT4 asym g128 reduce stage, INT8 asym g128 gather stage, fp16 output"),
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def outlier_channels(w: Workload, seed: int = 0) -> torch.Tensor:
    """The fixed set of hidden channels that carry the outlier gain (CPU)."""
    p = w.params
    if "n_chan" in p:
        k = p["n_chan"]
    elif "chan_frac" in p:
        k = max(1, int(round(p["chan_frac"] * w.cols)))
    else:
        return torch.zeros(0, dtype=torch.long)
    return torch.randperm(w.cols, generator=_gen("cpu", seed + 1000))[:k]


def step_factor(w: Workload, step: int, seed: int = 0) -> float:
    """Per-step magnitude drift factor exp(U[ln lo, ln hi]) (drawn on CPU)."""
    if w.dist != "normal_drift":
        return 1.0
    u = torch.rand((), generator=_gen("cpu", seed + 5000 + step), dtype=torch.float64).item()
    lo, hi = math.log(w.params["lo"]), math.log(w.params["hi"])
    return math.exp(lo + (hi - lo) * u)


def laplace_from_uniform(r: torch.Tensor, b: float) -> torch.Tensor:
    """Laplace(0, b) by the inverse CDF, evaluated at the cell midpoints
    (k + 1/2)/2^24 of float32 uniforms r = k/2^24, so |u| < 1/2 and every
    draw is finite (r = 0 would otherwise give -inf)."""
    u = (r.double() + 2.0 ** -25) - 0.5
    return (-b * torch.sign(u) * torch.log1p(-2.0 * u.abs())).float()


def rank_values_f32(w: Workload, rank: int, rows: int | None = None, cols: int | None = None,
                    seed: int = 0, device="cpu", step: int = 0) -> torch.Tensor:
    """float32 values of one rank's tensor before rounding to the 16-bit dtype."""
    rows = w.rows if rows is None else rows
    cols = w.cols if cols is None else cols
    g = _gen(device, seed + rank)
    p = w.params
    shape = (rows, cols)
    if w.dist == "mix_outlier":
        base = torch.randn(shape, generator=g, device=device) * p["sigma"]
        out = torch.randn(shape, generator=g, device=device) * p["sigma_out"]
        pick = torch.rand(shape, generator=g, device=device) < p["p_out"]
        x = torch.where(pick, out, base)
    elif w.dist == "laplace":
        x = laplace_from_uniform(torch.rand(shape, generator=g, device=device), p["b"])
    elif w.dist == "normal_drift":
        x = torch.randn(shape, generator=g, device=device) * (p["sigma"] * step_factor(w, step, seed))
    elif w.dist == "normal":
        x = torch.randn(shape, generator=g, device=device) * p["sigma"]
    elif w.dist == "student_t":
        z = torch.randn(shape, generator=g, device=device)
        chi2 = torch.zeros(shape, device=device)
        for _ in range(p["df"]):
            chi2 += torch.randn(shape, generator=g, device=device) ** 2
        x = z / torch.sqrt(chi2 / p["df"]) * p["scale"]
    else:
        raise ValueError(w.dist)
    ch = outlier_channels(w, seed)
    ch = ch[ch < cols]
    if ch.numel():
        x[:, ch.to(device)] *= p["chan_gain"]
    return x


def make_rank_inputs(w: Workload, rows: int | None = None, cols: int | None = None,
                     ranks: int | None = None, seed: int = 0, device="cpu",
                     step: int = 0) -> torch.Tensor:
    """[ranks, rows, cols] tensor in the workload's 16-bit dtype, contiguous."""
    rows = w.rows if rows is None else rows
    cols = w.cols if cols is None else cols
    ranks = w.ranks if ranks is None else ranks
    out = torch.empty((ranks, rows, cols), dtype=w.torch_dtype, device=device)
    for r in range(ranks):
        out[r] = rank_values_f32(w, r, rows, cols, seed, device, step).to(w.torch_dtype)
    return out
