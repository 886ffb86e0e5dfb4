"""Full-size parity: every workload at its full size, through the same calls
and launch configuration the benchmark times, checked against the oracle on
sampled rows (the oracle computes those rows from the inputs alone) and on
per-tensor quantities the oracle computes over whole tensors.

Step checked: compress all ranks (CURRENT mode for TACO, so the per-tensor
scale is a function of the data) -> dequantize-reduce all rows -> requantize
the sum for the gather stage (DELAYED, with a per-shard scale fixed by the
test) -> decompress."""
import multiprocessing as mp
import os

import numpy as np
import pytest
import torch

import oracle as orc
import oracle_pool
import quantized_tensor_activation_gb300 as qta
import workloads
from gpu_util import ORC_SCH, assert_close_f32, assert_same, bits, device

pytestmark = pytest.mark.gpu

N_SAMPLE_ROWS = 12


@pytest.fixture(scope="module")
def dev():
    return device()


@pytest.fixture(scope="module")
def pool():
    ctx = mp.get_context("spawn")
    p = ctx.Pool(max(1, min(8, (os.cpu_count() or 2) - 1)))
    yield p
    p.close()
    p.join()


def _oracle_k1_state(pool, xb, N, R, C, B):
    """The oracle's CURRENT-mode per-tensor state {S, amax} of every rank,
    over whole rank tensors (max |H x| gathered shard by shard)."""
    gr = R // N
    parts = pool.map(oracle_pool.rows_amax, [(np.ascontiguousarray(xb[:, j * gr:(j + 1) * gr]).reshape(-1),
                                              orc.BF16, N, gr, C, B) for j in range(N)])
    amax = np.max(np.array(parts, dtype=np.float32), axis=0)
    st = np.zeros(2 * N, dtype=np.float32)
    st[0::2] = [orc.scale_from_amax(a) for a in amax]
    st[1::2] = amax
    return st


def _oracle_gather_state(pool, xb, N, R, C, B, gB, st1, S2, fused):
    """The oracle's gather-stage state of every output shard (DELAYED, scale
    S2[j], amax over the whole shard), computed shard by shard."""
    gr = R // N
    tasks = [(np.ascontiguousarray(xb[:, j * gr:(j + 1) * gr]).reshape(-1), orc.BF16, N, gr, C, orc.TACO_FP8, B,
              list(st1[0::2]), orc.TACO_FP8, gB, [S2[2 * j], 0.0], orc.DELAYED, fused, [0], orc.BF16)
             for j in range(N)]
    res = pool.map(oracle_pool.shard_chain, tasks)
    return np.array([v for r in res for v in r["g_state"]], dtype=np.float32)


def _rows_of(buf: torch.Tensor, rows_idx, per_row: int) -> np.ndarray:
    """Bytes of the given rows of a flat byte buffer with per_row bytes/row."""
    b = buf.view(-1, per_row)[torch.as_tensor(rows_idx, device=buf.device)]
    return bits(b)


@pytest.mark.parametrize("name", ["taco_tiny", "gpt_tp", "qwen_grad", "equarx_int8", "flash_int4"])
def test_workload_full_size(dev, pool, name):
    w = workloads.WORKLOADS[name]
    N, R, C, B, gB = w.ranks, w.rows, w.cols, w.block, w.gather_block
    s1, s2 = qta.SCHEMES[w.scheme], qta.SCHEMES[w.gather_scheme]
    in_dt = qta.BF16 if w.dtype == "bf16" else qta.FP16
    o_dt = orc.BF16 if w.dtype == "bf16" else orc.FP16
    x = workloads.make_rank_inputs(w, device=dev, seed=7)

    # ---- the benchmark's calls
    d_in = qta.desc(s1, B, R, C, batch=N)
    q = qta.alloc_qtensor(d_in, dev)
    mode = qta.SCALE_CURRENT if s1 == qta.TACO_FP8 else qta.SCALE_DELAYED
    qta.taco_compress(d_in, x, in_dt, q, mode)
    d1 = qta.desc(s1, B, R, C)
    ssum = torch.empty((R, C), dtype=torch.float32, device=dev)
    qta.qar_reduce(d1, [q.shard(r) for r in range(N)], 0, R, ssum)
    gr = R // N
    d_g = qta.desc(s2, gB, gr, C, batch=N)
    g = qta.alloc_qtensor(d_g, dev)
    S2 = np.array([0.0, 0.0] * N, dtype=np.float32)
    S2[0::2] = [2.0 ** -7 * (1 + 0.25 * j) for j in range(N)]   # fixed gather-stage scales
    if g.state is not None:
        g.state.copy_(torch.from_numpy(S2))
    qta.qar_requant(d_g, ssum, g, qta.SCALE_DELAYED)
    y = torch.empty((R, C), dtype=w.torch_dtype, device=dev)
    qta.taco_decompress(d_g, g, y, in_dt)
    torch.cuda.synchronize()
    assert qta.qta_device_error() == 0

    # ---- per-tensor scales (TACO): the compress's in CURRENT mode and the
    # gather stage's (DELAYED with S2, amax over each whole output shard),
    # both from the oracle over whole tensors
    st = None
    if s1 == qta.TACO_FP8:
        xall = bits(x).reshape(N, R, C)
        st = _oracle_k1_state(pool, xall, N, R, C, B)
        assert_same("per-tensor state", q.state, st)
        if s2 == qta.TACO_FP8:
            assert in_dt == qta.BF16
            gst = _oracle_gather_state(pool, xall, N, R, C, B, gB, st, S2, fused=False)
            assert_same("gather-stage state", g.state, gst)
        del xall

    # ---- sampled rows
    rng = np.random.default_rng(hash(name) % 2 ** 32)
    rows = np.unique(np.concatenate([[0, R - 1, gr - 1, gr], rng.choice(R, N_SAMPLE_ROWS, replace=False)]))
    k = len(rows)
    xs = x[:, torch.as_tensor(rows, device=dev)].contiguous().cpu()              # [N, k, C]
    xb = bits(xs)
    cpr = C // 2 if s1 == qta.INT4_ASYM_G128 else C                              # code bytes per row
    ref = []
    for r in range(N):
        st_r = None if st is None else st[2 * r:2 * r + 2].copy()
        c, s, z = orc.compress(ORC_SCH[s1], B, xb[r * k * C:(r + 1) * k * C], o_dt, 1, k, C, st_r, orc.DELAYED)
        ref.append((c, s, z, st_r))
        # the GPU's codes / scales of those rows of rank r
        sh = q.shard(r)
        assert_same(f"rank {r} codes", _rows_of(sh.codes, rows, cpr), c)
        sbytes = {qta.TACO_FP8: 1, qta.INT8_SYM_B64: 4}.get(s1, 2) * (C // B)
        assert_same(f"rank {r} scales", _rows_of(sh.scales, rows, sbytes), s)
        if z is not None:
            assert_same(f"rank {r} zeros", _rows_of(sh.zeros, rows, sbytes), z)
    osum = orc.reduce(ORC_SCH[s1], B, ref, k, C)
    gsum = ssum[torch.as_tensor(rows, device=dev)]
    assert_same("sum rows", gsum, osum)
    assert_close_f32("sum rows", gsum, osum)

    # requant of the sampled rows: each row belongs to shard row // gr
    gcodes = []
    for i, row in enumerate(rows):
        j = row // gr
        stj = None if g.state is None else S2[2 * j:2 * j + 2].copy()
        c, s, z = orc.compress(ORC_SCH[s2], gB, osum[i * C:(i + 1) * C], orc.FP32, 1, 1, C, stj, orc.DELAYED)
        gcodes.append((c, s, z, stj))
    gcpr = C // 2 if s2 == qta.INT4_ASYM_G128 else C
    gsb = {qta.TACO_FP8: 1, qta.INT8_SYM_B64: 4}.get(s2, 2) * (C // gB)
    assert_same("requant codes", _rows_of(g.codes, rows, gcpr), np.concatenate([c[0] for c in gcodes]))
    assert_same("requant scales", _rows_of(g.scales, rows, gsb), np.concatenate([c[1] for c in gcodes]))
    if gcodes[0][2] is not None:
        assert_same("requant zeros", _rows_of(g.zeros, rows, gsb), np.concatenate([c[2] for c in gcodes]))
    yo = np.concatenate([orc.decompress(ORC_SCH[s2], gB, c, s, z, stj, 1, 1, C, o_dt) for c, s, z, stj in gcodes])
    assert_same("output rows", y[torch.as_tensor(rows, device=dev)], yo)


@pytest.mark.parametrize("name", ["taco_tiny", "gpt_tp", "qwen_grad", "equarx_int8", "flash_int4"])
def test_workload_full_size_fused_as_benched(dev, pool, name):
    """The timed step's own calls at full size: the compress on a capped SM
    count (as the benchmark may choose), the fused reduce + requant with the
    gather stage's per-shard DELAYED scales, the decompress; sampled rows
    against the oracle's fused function, row by row."""
    w = workloads.WORKLOADS[name]
    N, R, C, B, gB = w.ranks, w.rows, w.cols, w.block, w.gather_block
    s1, s2 = qta.SCHEMES[w.scheme], qta.SCHEMES[w.gather_scheme]
    in_dt = qta.BF16 if w.dtype == "bf16" else qta.FP16
    o_dt = orc.BF16 if w.dtype == "bf16" else orc.FP16
    x = workloads.make_rank_inputs(w, device=dev, seed=11)

    d_in = qta.desc(s1, B, R, C, batch=N, max_sms=144)
    q = qta.alloc_qtensor(d_in, dev)
    qta.taco_compress(d_in, x, in_dt, q, qta.SCALE_CURRENT if s1 == qta.TACO_FP8 else qta.SCALE_DELAYED)
    gr = R // N
    d_sh = qta.desc(s1, B, R, C)
    d_g = qta.desc(s2, gB, gr, C, batch=N)
    g = qta.alloc_qtensor(d_g, dev)
    S2 = np.zeros(2 * N, dtype=np.float32)
    S2[0::2] = [2.0 ** -7 * (1 + 0.25 * j) for j in range(N)]
    if g.state is not None:
        g.state.copy_(torch.from_numpy(S2))
    qta.qar_reduce_requant(d_sh, [q.shard(r) for r in range(N)], 0, R, d_g, g, qta.SCALE_DELAYED)
    y = torch.empty((R, C), dtype=w.torch_dtype, device=dev)
    qta.taco_decompress(d_g, g, y, in_dt)
    torch.cuda.synchronize()
    assert qta.qta_device_error() == 0

    rng = np.random.default_rng(hash(name) % 2 ** 31 + 1)
    rows = np.unique(np.concatenate([[0, R - 1, gr - 1, gr], rng.choice(R, 8, replace=False)]))
    k = len(rows)
    xb = bits(x[:, torch.as_tensor(rows, device=dev)].contiguous().cpu())
    st = None
    if s1 == qta.TACO_FP8:
        xall = bits(x).reshape(N, R, C)
        st = _oracle_k1_state(pool, xall, N, R, C, B)
        assert_same("per-tensor state", q.state, st)
        if s2 == qta.TACO_FP8:
            gst = _oracle_gather_state(pool, xall, N, R, C, B, gB, st, S2, fused=True)
            assert_same("gather-stage state", g.state, gst)
        del xall
    shards = []
    for r in range(N):
        st_r = None if st is None else st[2 * r:2 * r + 2].copy()
        c, s, z = orc.compress(ORC_SCH[s1], B, xb[r * k * C:(r + 1) * k * C], o_dt, 1, k, C, st_r, orc.DELAYED)
        shards.append((c, s, z, st_r))
    gcpr = C // 2 if s2 == qta.INT4_ASYM_G128 else C
    gsb = {qta.TACO_FP8: 1, qta.INT8_SYM_B64: 4}.get(s2, 2) * (C // gB)
    want_c, want_s, want_z, want_y = [], [], [], []
    for i, row in enumerate(rows):
        j = row // gr
        stj = None if g.state is None else np.array([S2[2 * j], 0.0], dtype=np.float32)
        c, s, z = orc.reduce_requant(ORC_SCH[s1], B, shards, k, C, i, i + 1, ORC_SCH[s2], gB, 1, stj, orc.DELAYED)
        want_c.append(c)
        want_s.append(s)
        want_z.append(z)
        want_y.append(orc.decompress(ORC_SCH[s2], gB, c, s, z, stj, 1, 1, C, o_dt))
    assert_same("fused codes", _rows_of(g.codes, rows, gcpr), np.concatenate(want_c))
    assert_same("fused scales", _rows_of(g.scales, rows, gsb), np.concatenate(want_s))
    if want_z[0] is not None:
        assert_same("fused zeros", _rows_of(g.zeros, rows, gsb), np.concatenate(want_z))
    assert_same("output rows", y[torch.as_tensor(rows, device=dev)], np.concatenate(want_y))
