"""Per-tensor choice of the Hadamard block size by reconstruction error: the
data-driven reshape of TACO (review page, Core claim: the reshape of the
intermediate tensor before the Adaptive Scale-Hadamard transform is chosen
from the data; no rule is printed).  Each candidate B is tried on the tensor
through the library itself -- taco_compress (CURRENT scale), taco_decompress
to FP32 and qta_sq_error -- and the block size with the smallest squared
error wins (the smaller B on a tie)."""
from __future__ import annotations

import torch

from . import BF16, FP16, FP32, SCALE_CURRENT, alloc_qtensor, desc, qta_sq_error, taco_compress, taco_decompress

_DT = {torch.bfloat16: BF16, torch.float16: FP16, torch.float32: FP32}


def block_errors(x: torch.Tensor, candidates=(64, 128, 256), mode: int = SCALE_CURRENT) -> dict:
    """x: device [rows, cols] or [batch, rows, cols] (bf16, fp16 or fp32).
    Returns {B: sum of squared reconstruction errors} for every candidate
    that divides cols."""
    if x.dim() == 2:
        x = x.unsqueeze(0)
    batch, rows, cols = x.shape
    x = x.contiguous()
    dt = _DT[x.dtype]
    y = torch.empty(x.shape, dtype=torch.float32, device=x.device)
    out = torch.empty(1, dtype=torch.float64, device=x.device)
    errs = {}
    for B in candidates:
        if cols % B:
            continue
        d = desc("taco_fp8", B, rows, cols, batch=batch)
        q = alloc_qtensor(d, x.device)
        taco_compress(d, x, dt, q, mode)
        taco_decompress(d, q, y, FP32)
        qta_sq_error(x, dt, y, x.numel(), out)
        errs[B] = float(out.item())
    return errs


def choose_block(x: torch.Tensor, candidates=(64, 128, 256), mode: int = SCALE_CURRENT):
    """(best block size, {B: squared error})."""
    errs = block_errors(x, candidates, mode)
    if not errs:
        raise ValueError("no candidate block size divides the number of columns")
    best = min(sorted(errs), key=lambda b: errs[b])
    return best, errs
