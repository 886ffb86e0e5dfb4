"""The oracle's work on a full-size workload, split by output shard, for the
full-size GPU tests.  Test infrastructure: run in worker processes of a
``spawn`` pool (so no worker is forked from a process that holds a CUDA
context), each task computes one output shard's rows from the input rows of
that shard alone.

Shard j of the gather stage holds rows [j R/N, (j+1) R/N) of the reduced
tensor; every step of the path is row-local except the per-tensor amax of
the compress (whole rank tensors), which a task takes as its input scale
(DELAYED) and returns as the amax over its rows, so that the caller can
combine it across shards.
"""
from __future__ import annotations

import numpy as np

import oracle as orc


def rows_amax(task):
    """Per-rank max |H x| (TACO, block B) over the given rows: the amax a
    CURRENT-mode compress of the whole tensor takes the max of."""
    xbits, dtype, n, k, cols, B = task
    out = []
    for r in range(n):
        x = xbits[r * k * cols:(r + 1) * k * cols]
        xf = orc.bf16_to_f32(x) if dtype == orc.BF16 else (orc.f16_to_f32(x) if dtype == orc.FP16 else x)
        out.append(float(np.abs(orc.fwht(xf, B)).max()) if x.size else 0.0)
    return out


def _rows(a, per_row, idx):
    a = np.asarray(a).reshape(-1, per_row)
    return a[idx].reshape(-1).copy()


def shard_chain(task):
    """One gather shard of one step: compress the shard's rows of every rank
    (DELAYED, with the ranks' per-tensor scales S1), reduce them, requantize
    the sum for the gather stage (fused: orc.reduce_requant; split: orc.reduce
    then orc.compress of the FP32 rows) with this shard's gather state, and
    decompress.  Returns the per-rank amax over the rows, the gather state,
    and the sampled rows (local indices) of every output."""
    (xbits, dtype, n, k, cols, s1, B, S1, s2, gB, g_state, g_mode, fused, sample, out_dtype) = task
    st1 = None
    if s1 == orc.TACO_FP8:
        st1 = np.zeros(2 * n, dtype=np.float32)
        st1[0::2] = S1
    c, s, z = orc.compress(s1, B, xbits, dtype, n, k, cols, st1, orc.DELAYED)
    E = k * cols
    cb = orc.codes_nbytes(s1, E)
    nb = E // B
    shards = [(c[r * cb:(r + 1) * cb], s[r * nb:(r + 1) * nb], None if z is None else z[r * nb:(r + 1) * nb],
               None if st1 is None else st1[2 * r:2 * r + 2]) for r in range(n)]
    gst = None if g_state is None else np.array(g_state, dtype=np.float32)
    if fused:
        oc, os_, oz = orc.reduce_requant(s1, B, shards, k, cols, 0, k, s2, gB, 1, gst, g_mode)
        ssum = None
    else:
        ssum = orc.reduce(s1, B, shards, k, cols)
        oc, os_, oz = orc.compress(s2, gB, ssum, orc.FP32, 1, k, cols, gst, g_mode)
    y = orc.decompress(s2, gB, oc, os_, oz, gst, 1, k, cols, out_dtype)
    sample = np.asarray(sample, dtype=np.int64)
    cpr = cb // k
    spr = s.nbytes // n // k
    k1 = []
    for r in range(n):
        sh = shards[r]
        k1.append((_rows(sh[0], cpr, sample), _rows(sh[1].view(np.uint8), spr, sample),
                   None if sh[2] is None else _rows(sh[2].view(np.uint8), spr, sample)))
    gcpr = oc.size // k
    gspr = os_.nbytes // k
    return {
        "k1_amax": None if st1 is None else [float(v) for v in st1[1::2]],
        "g_state": None if gst is None else [float(v) for v in gst],
        "k1_rows": k1,
        "sum_rows": None if ssum is None else _rows(ssum, cols, sample),
        "g_codes": _rows(oc.view(np.uint8), gcpr, sample),
        "g_scales": _rows(os_.view(np.uint8), gspr, sample),
        "g_zeros": None if oz is None else _rows(oz.view(np.uint8), gspr, sample),
        "y_rows": _rows(y, cols, sample),
    }
