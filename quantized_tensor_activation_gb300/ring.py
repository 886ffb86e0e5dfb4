"""Quantized ring reduce-scatter / all-reduce of n simulated ranks, as the
adder chains of EQuARX (review page, Figs. 4-5: full-loop and semi-loop
adder chains; What carries the argument: each received partial sum is
dequantized to FP32 before the receiver adds its own shard, and the sum is
requantized before it travels on).

Every arithmetic step is a call of the C ABI (taco_compress,
qar_dequant_add_requant, qar_dequant_add, qar_requant, taco_decompress);
this module only sequences the hops and holds the buffers.  Chunk j (rows
j*R/n .. (j+1)*R/n of every rank's [R, C] tensor) is owned by rank j.
  full loop: one chain j+1, j+2, ..., j+n-1, then the owner;
  semi loop: two chains that meet at the owner, j+h, ..., j+1 and
             j-(n-1-h), ..., j-1, with h = n // 2.
The first rank of a chain quantizes its chunk; each following rank
dequantizes the incoming partial sum, adds its chunk and requantizes (scale
mode CURRENT for TACO: the magnitude grows along the chain); the owner adds
its own chunk to the first chain's partial sum, then the second chain's.
"""
from __future__ import annotations

import torch

from . import (BF16, FP16, FP32, SCALE_CURRENT, Desc, alloc_qtensor, desc, qar_dequant_add,
               qar_dequant_add_requant, qar_requant, taco_compress, taco_decompress)

_DT = {torch.bfloat16: BF16, torch.float16: FP16, torch.float32: FP32}


def chunk_orders(n: int, j: int, semi: bool):
    """Visiting orders of the chains that end at the owner j."""
    if not semi:
        return [[(j + k) % n for k in range(1, n)]]
    h = n // 2
    chains = [[(j + k) % n for k in range(h, 0, -1)]]
    if n - 1 - h > 0:
        chains.append([(j - k) % n for k in range(n - 1 - h, 0, -1)])
    return chains


def _alloc_stream(stream, dev):
    """The stream the ring's work runs on, as a torch stream (a raw handle
    or None means the current stream)."""
    return stream if isinstance(stream, torch.cuda.Stream) else torch.cuda.current_stream(dev)


def _chunk_desc(d: Desc, n: int) -> Desc:
    if n < 2:
        raise ValueError("a ring needs at least two ranks")
    if d.batch != 1 or d.rows % n:
        raise ValueError("the ring takes one [rows, cols] tensor per rank with rows divisible by the ranks")
    return desc(d.scheme, d.block, d.rows // n, d.cols, max_sms=d.max_sms)


def reduce_scatter(d: Desc, xs: torch.Tensor, semi: bool = False, hop_partials: list | None = None,
                   stream=None) -> torch.Tensor:
    """xs: [n, rows, cols] device tensor (bf16, fp16 or fp32), the ranks'
    inputs; d: scheme, block and [rows, cols] of one rank.  Returns the FP32
    reduce-scatter result [rows, cols] (chunk j = the sum owned by rank j).
    If hop_partials is a list, the full loop appends after every hop k the
    dequantized partial sums of all chunks ([rows, cols] FP32)."""
    n = xs.shape[0]
    dc = _chunk_desc(d, n)
    rc = dc.rows
    dt = _DT[xs.dtype]
    dev = xs.device
    # the buffers are allocated on the stream that uses them, so that the
    # caching allocator orders their reuse after this work
    with torch.cuda.stream(_alloc_stream(stream, dev)):
        out = torch.empty((d.rows, d.cols), dtype=torch.float32, device=dev)
        tmp = torch.empty((rc, d.cols), dtype=torch.float32, device=dev)
        bufs = [[alloc_qtensor(dc, dev), alloc_qtensor(dc, dev)] for _ in range(2)]

    def chunk(r, j):
        return xs[r, j * rc:(j + 1) * rc]

    rec = hop_partials is not None and not semi
    if rec:
        for _ in range(n - 1):
            hop_partials.append(torch.empty((d.rows, d.cols), dtype=torch.float32, device=dev))
    for j in range(n):
        finals = []
        for c, order in enumerate(chunk_orders(n, j, semi)):
            a, b = bufs[c]
            taco_compress(dc, chunk(order[0], j), dt, a, SCALE_CURRENT, stream)
            if rec:
                taco_decompress(dc, a, hop_partials[0][j * rc:(j + 1) * rc], FP32, stream)
            for k, r in enumerate(order[1:], start=1):
                qar_dequant_add_requant(dc, a, chunk(r, j), dt, b, SCALE_CURRENT, stream)
                a, b = b, a
                if rec:
                    taco_decompress(dc, a, hop_partials[k][j * rc:(j + 1) * rc], FP32, stream)
            finals.append(a)
        dst = out[j * rc:(j + 1) * rc]
        if len(finals) == 1:
            qar_dequant_add(dc, finals[0], chunk(j, j), dt, dst, stream)
        else:
            qar_dequant_add(dc, finals[0], chunk(j, j), dt, tmp, stream)
            qar_dequant_add(dc, finals[1], tmp, FP32, dst, stream)
    return out


def allreduce(d: Desc, xs: torch.Tensor, semi: bool = False, out_dtype=torch.float32, stream=None):
    """Ring reduce-scatter, then the quantized all-gather: each reduced chunk
    is requantized (CURRENT scale for TACO) and dequantized by every rank.
    Returns (reduce-scatter FP32 sums, all-reduce output in out_dtype)."""
    n = xs.shape[0]
    s = reduce_scatter(d, xs, semi, stream=stream)
    dc = _chunk_desc(d, n)
    rc = dc.rows
    with torch.cuda.stream(_alloc_stream(stream, xs.device)):
        g = alloc_qtensor(dc, xs.device)
        y = torch.empty((d.rows, d.cols), dtype=out_dtype, device=xs.device)
    for j in range(n):
        qar_requant(dc, s[j * rc:(j + 1) * rc], g, SCALE_CURRENT, stream)
        taco_decompress(dc, g, y[j * rc:(j + 1) * rc], _DT[out_dtype], stream)
    return s, y
