"""GPU parity on paths the other tests leave out:

* the tie rule on the GPU: inputs whose scaled value is exactly k + 1/2 give
  the even code (reading: every rounding is round-to-nearest-even), through
  the compress (16-bit and FP32 inputs, i.e. also the requantizer);
* more tensors than a CTA's shared-memory amax table holds (64): tensors
  64 .. 79 of a batch take the global atomicMax path of the per-tensor amax
  -- in the compress (both scale modes), the fused reduce + requant with 80
  output shards, and the requantizing ring hop; the state is compared bit
  for bit;
* the Qwen-style gradient workload as specified: 16 successive steps at full
  size, each with its own log-uniform magnitude factor, step 0 CURRENT and
  the later ones DELAYED with the scales taco_update_scale left (TACO Core
  claim: stability across training steps); every step's per-tensor states
  of both stages are compared with the oracle's over whole tensors, and
  sampled rows of every output bit for bit;
* INT4 groups at the edges of the reduce's scaled decode (terms and partial
  sums formed scaled by 2^-24 / 2^-20, the sum scaled back at the end):
  zero-points far below the scale, minima exactly 0, constant groups (s = 0)
  and groups of fp16 subnormals (subnormal scale and zero-point), through
  the FP32 reduce, the fused reduce + INT8 requant and the decompress.
"""
import multiprocessing as mp
import os

import numpy as np
import pytest
import torch

import oracle as orc
import oracle_pool
import quantized_tensor_activation_gb300 as qta
import workloads
from gpu_util import (ORC_SCH, assert_same, bits, compare_qtensor, device, gpu_compress, oracle_bits_in,
                      oracle_compress, random_values, to_dtype_cpu)

pytestmark = pytest.mark.gpu


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


# ------------------------------------------------------------------ ties
def _int8_tie_input():
    k = np.array([0, 1, 2, 3, 10, 125, -1, -2, -3, -126, 62, 63, 64, 99, 100, -100], dtype=np.float64)
    blocks = []
    for b in (np.concatenate([k + 0.5, [127.0]]), np.concatenate([2 * k + 1, [254.0]])):
        x = np.zeros(64)
        x[:b.size] = b
        blocks.append(x)
    want = np.array([int(2 * np.round((kk + 0.5) / 2)) for kk in k])     # the even neighbour of k + 1/2
    return np.concatenate(blocks * 32).astype(np.float32).reshape(8, 512), k.size, want


@pytest.mark.parametrize("dtype", [qta.BF16, qta.FP32])
def test_int8_sym_ties_to_even_on_gpu(dev, dtype):
    x, nk, want = _int8_tie_input()
    xt = to_dtype_cpu(x, dtype)
    assert np.array_equal(xt.float().numpy(), x)
    _, q = gpu_compress(qta.INT8_SYM_B64, 64, xt.reshape(1, 8, 512), dtype, 1, 8, 512, dev=dev)
    ref = oracle_compress(qta.INT8_SYM_B64, 64, xt, dtype, 1, 8, 512)
    torch.cuda.synchronize()
    compare_qtensor("int8 ties", q, ref)
    c = q.codes.cpu().numpy().view(np.int8).reshape(-1, 64).astype(np.int64)
    for blk in range(c.shape[0]):
        assert np.array_equal(c[blk, :nk], want), blk


@pytest.mark.parametrize("bits_", [4, 8])
@pytest.mark.parametrize("dtype", [qta.FP16, qta.FP32])
@pytest.mark.parametrize("zero", [0.0, -1.0, 3.5])
def test_asym_ties_to_even_on_gpu(dev, bits_, dtype, zero):
    Q = 2 ** bits_ - 1
    s = 0.125 if bits_ == 8 else 0.25
    scheme = qta.INT8_ASYM_G128 if bits_ == 8 else qta.INT4_ASYM_G128
    ks = np.resize(np.arange(Q), 126)
    g = np.concatenate([[zero, zero + Q * s], zero + (ks + 0.5) * s])
    x = np.tile(g, 24).astype(np.float32).reshape(6, 512)
    xt = to_dtype_cpu(x, dtype)
    assert np.array_equal(xt.float().numpy(), x)
    _, q = gpu_compress(scheme, 128, xt.reshape(1, 6, 512), dtype, 1, 6, 512, dev=dev)
    ref = oracle_compress(scheme, 128, xt, dtype, 1, 6, 512)
    torch.cuda.synchronize()
    compare_qtensor("asym ties", q, ref)
    c = q.codes.cpu().numpy()
    qq = c if bits_ == 8 else np.stack([c & 15, c >> 4], axis=1).reshape(-1)
    qq = qq.reshape(-1, 128).astype(np.int64)
    want = 2 * np.round((ks + 0.5) / 2).astype(np.int64)
    assert np.all(qq[:, 0] == 0) and np.all(qq[:, 1] == Q)
    assert np.all(qq[:, 2:] == want[None, :])


# ------------------------------------------------------------------ > 64 tensors
N_TENSORS = 80


@pytest.mark.parametrize("mode", [qta.SCALE_CURRENT, qta.SCALE_DELAYED])
@pytest.mark.parametrize("B", [128, 256])
def test_taco_compress_80_tensors(dev, mode, B):
    rows, cols = 3, 512                      # 24 segments per tensor: tensors share warp tiles
    rng = np.random.default_rng(B + mode)
    x = random_values(rng, (N_TENSORS, rows, cols), "mixed")
    x *= np.exp(rng.uniform(-3, 3, (N_TENSORS, 1, 1))).astype(np.float32)
    xt = to_dtype_cpu(x, qta.BF16)
    state = np.zeros(2 * N_TENSORS, dtype=np.float32)
    state[0::2] = np.exp(rng.uniform(-6, 0, N_TENSORS)).astype(np.float32)
    state[1::2] = np.where(np.arange(N_TENSORS) % 3 == 0, 0.5, 0.0).astype(np.float32)
    _, q = gpu_compress(qta.TACO_FP8, B, xt, qta.BF16, N_TENSORS, rows, cols, mode, state=state, dev=dev)
    ref = oracle_compress(qta.TACO_FP8, B, xt, qta.BF16, N_TENSORS, rows, cols,
                          orc.CURRENT if mode == qta.SCALE_CURRENT else orc.DELAYED, state=state)
    torch.cuda.synchronize()
    compare_qtensor("80 tensors", q, ref)
    assert qta.qta_device_error() == 0


@pytest.mark.parametrize("mode", [qta.SCALE_CURRENT, qta.SCALE_DELAYED])
def test_reduce_requant_80_output_shards(dev, mode):
    B, n, rows, cols = 128, 3, 2 * N_TENSORS, 768     # 24 segments per output shard
    rng = np.random.default_rng(5 + mode)
    xt = to_dtype_cpu(random_values(rng, (n, rows, cols), "laplace"), qta.BF16)
    d, q = gpu_compress(qta.TACO_FP8, B, xt, qta.BF16, n, rows, cols, dev=dev)
    ref = oracle_compress(qta.TACO_FP8, B, xt, qta.BF16, n, rows, cols)
    E, nb = rows * cols, rows * cols // B
    shards = [(ref[0][r * E:(r + 1) * E], ref[1][r * nb:(r + 1) * nb], None, ref[3][2 * r:2 * r + 2])
              for r in range(n)]
    dg = qta.desc(qta.TACO_FP8, B, rows // N_TENSORS, cols, batch=N_TENSORS)
    g = qta.alloc_qtensor(dg, dev)
    gst = np.zeros(2 * N_TENSORS, dtype=np.float32)
    gst[0::2] = np.exp(rng.uniform(-7, -3, N_TENSORS)).astype(np.float32)
    g.state.copy_(torch.from_numpy(gst))
    d1 = qta.desc(qta.TACO_FP8, B, rows, cols)
    qta.qar_reduce_requant(d1, [q.shard(r) for r in range(n)], 0, rows, dg, g, mode)
    oc, os_, _ = orc.reduce_requant(orc.TACO_FP8, B, shards, rows, cols, 0, rows, orc.TACO_FP8, B, N_TENSORS,
                                    gst, orc.CURRENT if mode == qta.SCALE_CURRENT else orc.DELAYED)
    torch.cuda.synchronize()
    compare_qtensor("stage 1", q, ref)
    assert_same("80 shards codes", g.codes, oc)
    assert_same("80 shards scales", g.scales, os_)
    assert_same("80 shards state", g.state, gst)
    assert qta.qta_device_error() == 0


def test_ring_hop_requant_80_tensors(dev):
    B, rows, cols = 128, 2, 1024
    rng = np.random.default_rng(77)
    xin = to_dtype_cpu(random_values(rng, (N_TENSORS, rows, cols), "laplace"), qta.BF16)
    xloc = to_dtype_cpu(random_values(rng, (N_TENSORS, rows, cols), "laplace"), qta.BF16)
    d, qin = gpu_compress(qta.TACO_FP8, B, xin, qta.BF16, N_TENSORS, rows, cols, dev=dev)
    rin = oracle_compress(qta.TACO_FP8, B, xin, qta.BF16, N_TENSORS, rows, cols)
    out = qta.alloc_qtensor(d, dev)
    ost = np.zeros(2 * N_TENSORS, dtype=np.float32)
    ost[0::2] = np.exp(rng.uniform(-6, -2, N_TENSORS)).astype(np.float32)
    out.state.copy_(torch.from_numpy(ost))
    qta.qar_dequant_add_requant(d, qin, xloc.to(dev), qta.BF16, out, qta.SCALE_DELAYED)
    s = orc.dequant_add(orc.TACO_FP8, B, *rin, N_TENSORS, rows, cols, oracle_bits_in(xloc), orc.BF16)
    oc, os_, _ = orc.compress(orc.TACO_FP8, B, s, orc.FP32, N_TENSORS, rows, cols, ost, orc.DELAYED)
    torch.cuda.synchronize()
    assert_same("hop codes", out.codes, oc)
    assert_same("hop scales", out.scales, os_)
    assert_same("hop state", out.state, ost)
    assert qta.qta_device_error() == 0


# ------------------------------------------------------------------ 16-step drift
def _rows_of(buf: torch.Tensor, idx, per_row: int) -> np.ndarray:
    return bits(buf.view(-1, per_row)[torch.as_tensor(idx, device=buf.device)])


def test_qwen_grad_16_steps_full_size(dev, pool):
    w = workloads.WORKLOADS["qwen_grad"]
    N, R, C, B, gB = w.ranks, w.rows, w.cols, w.block, w.gather_block
    assert w.steps == 16
    gr = R // N
    d_in = qta.desc(qta.TACO_FP8, B, R, C, batch=N)
    d_sh = qta.desc(qta.TACO_FP8, B, R, C)
    d_g = qta.desc(qta.TACO_FP8, gB, gr, C, batch=N)
    q = qta.alloc_qtensor(d_in, dev)
    g = qta.alloc_qtensor(d_g, dev)
    shards = [q.shard(r) for r in range(N)]
    y = torch.empty((R, C), dtype=torch.bfloat16, device=dev)
    rng = np.random.default_rng(2)
    sample = np.unique(np.concatenate([[0, gr - 1, gr, R - 1], rng.choice(R, 6, replace=False)]))
    S1 = None                                 # the oracle's per-tensor scales of the compress
    Sg = [None] * N                           # and of the gather stage, per shard
    factors = set()
    for step in range(w.steps):
        factors.add(workloads.step_factor(w, step))
        x = workloads.make_rank_inputs(w, step=step)          # CPU bytes, handed to both sides
        xb = bits(x).reshape(N, R, C)
        mode = qta.SCALE_CURRENT if step == 0 else qta.SCALE_DELAYED
        # ---- GPU: the step as the benchmark runs it
        qta.taco_compress(d_in, x.to(dev), qta.BF16, q, mode)
        qta.qar_reduce_requant(d_sh, shards, 0, R, d_g, g, mode)
        qta.taco_decompress(d_g, g, y, qta.BF16)
        torch.cuda.synchronize()
        st1 = bits(q.state).view(np.float32).copy()
        stg = bits(g.state).view(np.float32).copy()
        k1 = [(_rows_of(sh.codes, sample, C), _rows_of(sh.scales, sample, C // B)) for sh in shards]
        gc = _rows_of(g.codes, sample, C)
        gs = _rows_of(g.scales, sample, C // gB)
        yr = bits(y[torch.as_tensor(sample, device=dev)])
        qta.taco_update_scale(q.state, N)
        qta.taco_update_scale(g.state, N)
        # ---- oracle, shard by shard
        if step == 0:
            parts = pool.map(oracle_pool.rows_amax, [(np.ascontiguousarray(xb[:, j * gr:(j + 1) * gr]).reshape(-1),
                                                      orc.BF16, N, gr, C, B) for j in range(N)])
            amax0 = np.max(np.array(parts, dtype=np.float32), axis=0)
            S1 = [orc.scale_from_amax(a) for a in amax0]
        tasks = []
        for j in range(N):
            loc = sample[(sample >= j * gr) & (sample < (j + 1) * gr)] - j * gr
            g_state = [1.0, 0.0] if step == 0 else [Sg[j], 0.0]
            tasks.append((np.ascontiguousarray(xb[:, j * gr:(j + 1) * gr]).reshape(-1), orc.BF16, N, gr, C,
                          orc.TACO_FP8, B, S1, orc.TACO_FP8, gB, g_state,
                          orc.CURRENT if step == 0 else orc.DELAYED, True, loc, orc.BF16))
        res = pool.map(oracle_pool.shard_chain, tasks)
        amax1 = np.max(np.array([r["k1_amax"] for r in res], dtype=np.float32), axis=0)
        want1 = np.zeros(2 * N, dtype=np.float32)
        want1[0::2] = S1
        want1[1::2] = amax1
        assert_same(f"step {step} compress state", st1, want1)
        wantg = np.array([v for r in res for v in r["g_state"]], dtype=np.float32)
        assert_same(f"step {step} gather state", stg, wantg)
        for r in range(N):
            assert_same(f"step {step} rank {r} codes", k1[r][0],
                        np.concatenate([res[j]["k1_rows"][r][0] for j in range(N)]))
            assert_same(f"step {step} rank {r} scales", k1[r][1],
                        np.concatenate([res[j]["k1_rows"][r][1] for j in range(N)]))
        assert_same(f"step {step} gather codes", gc, np.concatenate([r_["g_codes"] for r_ in res]))
        assert_same(f"step {step} gather scales", gs, np.concatenate([r_["g_scales"] for r_ in res]))
        assert_same(f"step {step} output rows", yr, np.concatenate([r_["y_rows"] for r_ in res]))
        # the next step's scales: S = amax/448 of this step (taco_update_scale)
        S1 = [orc.scale_from_amax(a) for a in amax1]
        Sg = [orc.scale_from_amax(wantg[2 * j + 1]) for j in range(N)]
        del x, xb, res, tasks
    assert len(factors) == w.steps and min(factors) >= 0.25 and max(factors) <= 4.0
    torch.cuda.synchronize()
    assert_same("final compress state", q.state, np.stack([np.array(S1, np.float32),
                                                            np.zeros(N, np.float32)], axis=1).reshape(-1))
    assert qta.qta_device_error() == 0


# ------------------------------------------------------------------ tiny per-tensor scales
@pytest.mark.parametrize("B", [64, 128, 256])
def test_tiny_per_tensor_scales(dev, B):
    # Per-tensor scales far below the usual range (2^-83 and 2^-100, with
    # inputs of that size) next to an ordinary one, with tensor boundaries
    # inside warp tiles: the decompress and the FP32 reduce must give the
    # oracle's bits (every multiply by 1/B and by the block scale keeps its
    # own rounding, also near the subnormal range).  The fourth tensor's
    # block scales lie near 2^-78, between the two.
    batch, rows, cols = 4, 11, 768
    rng = np.random.default_rng(B)
    x = random_values(rng, (batch, rows, cols), "mixed")
    x[0] *= np.float32(2.0 ** -75)
    x[2] *= np.float32(2.0 ** -92)
    x[3] *= np.float32(2.0 ** -70)
    xt = torch.from_numpy(x.astype(np.float32))
    state = np.array([2.0 ** -83, 0.0, 0.01, 0.0, 2.0 ** -100, 0.0, 2.0 ** -79, 0.0], dtype=np.float32)
    d, q = gpu_compress(qta.TACO_FP8, B, xt, qta.FP32, batch, rows, cols, qta.SCALE_DELAYED, state=state, dev=dev)
    ref = oracle_compress(qta.TACO_FP8, B, xt, qta.FP32, batch, rows, cols, orc.DELAYED, state=state)
    torch.cuda.synchronize()
    compare_qtensor("tiny S", q, ref)
    for od, tdt in ((qta.FP32, torch.float32), (qta.BF16, torch.bfloat16)):
        y = torch.empty((batch, rows, cols), dtype=tdt, device=dev)
        qta.taco_decompress(d, q, y, od)
        yo = orc.decompress(orc.TACO_FP8, B, *ref, batch, rows, cols, orc.FP32 if od == qta.FP32 else orc.BF16)
        torch.cuda.synchronize()
        assert_same(f"decompress {od}", y, yo)
    E, nb = rows * cols, rows * cols // B
    shards = [(ref[0][r * E:(r + 1) * E], ref[1][r * nb:(r + 1) * nb], None, ref[3][2 * r:2 * r + 2])
              for r in range(batch)]
    d1 = qta.desc(qta.TACO_FP8, B, rows, cols)
    for sel in ([0, 1, 2], [1], [0], [1, 2]):
        s = torch.empty((rows, cols), dtype=torch.float32, device=dev)
        qta.qar_reduce(d1, [q.shard(r) for r in sel], 0, rows, s)
        so = orc.reduce(orc.TACO_FP8, B, [shards[r] for r in sel], rows, cols)
        torch.cuda.synchronize()
        assert_same(f"reduce {sel}", s, so)
    assert qta.qta_device_error() == 0


def _int4_edge_data(rng, rows, cols):
    """Rows of 128-groups: N(0, 1) groups, and on every eighth row from row 3
    groups in [1e-6, 1] (an fp16-subnormal zero-point far below the scale),
    groups with minimum exactly 0, constant groups (s = 0) and groups in
    [0, 1e-6] (fp16 subnormals: subnormal scale and zero-point)."""
    x = rng.standard_normal((rows, cols)).astype(np.float32)
    g = x.reshape(rows, cols // 128, 128)
    for r in range(3, rows, 8):
        g[r, 0::4] = rng.uniform(0.0, 1.0, g[r, 0::4].shape)
        g[r, 0::4, 0] = 1e-6
        g[r, 1::4] = np.abs(g[r, 1::4])
        g[r, 1::4, 5] = 0.0
        g[r, 2::4] = 0.75
        g[r, 3::4] = rng.uniform(0.0, 1e-6, g[r, 3::4].shape)
    return x


def test_int4_edge_groups(dev):
    rows, cols, n = 256, 1024, 3
    rng = np.random.default_rng(41)
    shards, dsh = [], []
    d = qta.desc(qta.INT4_ASYM_G128, 128, rows, cols)
    for r in range(n):
        xt = to_dtype_cpu(_int4_edge_data(rng, rows, cols) * (1.0 + r), qta.FP16)
        c, s_, z, st = oracle_compress(qta.INT4_ASYM_G128, 128, xt, qta.FP16, 1, rows, cols)
        shards.append((c, s_, z, st))
        dsh.append(qta.QTensor(d, torch.from_numpy(c.view(np.uint8).copy()).to(dev),
                               torch.from_numpy(s_.view(np.uint8).copy()).to(dev),
                               torch.from_numpy(z.view(np.uint8).copy()).to(dev), None))
    # the data has the edge groups: subnormal fp16 scales and zero-points,
    # zero scales, zero zero-points
    s0 = shards[0][1].view(np.float16)
    z0 = shards[0][2].view(np.float16)
    tiny = np.float16(2.0 ** -14)
    assert ((s0 > 0) & (s0 < tiny)).any() and ((z0 > 0) & (z0 < tiny)).any()
    assert (s0 == 0).any() and (z0 == 0).any()

    out = torch.empty((rows, cols), dtype=torch.float32, device=dev)
    qta.qar_reduce(d, dsh, 0, rows, out)
    ref = orc.reduce(orc.INT4_ASYM, 128, shards, rows, cols)
    torch.cuda.synchronize()
    assert_same("int4 reduce, edge groups", out, ref)

    nb = 4
    dg = qta.desc(qta.INT8_ASYM_G128, 128, rows // nb, cols, batch=nb)
    g = qta.alloc_qtensor(dg, dev)
    qta.qar_reduce_requant(d, dsh, 0, rows, dg, g, qta.SCALE_CURRENT)
    c, s_, z = orc.reduce_requant(orc.INT4_ASYM, 128, shards, rows, cols, 0, rows, orc.INT8_ASYM, 128, nb, None,
                                  orc.CURRENT)
    torch.cuda.synchronize()
    compare_qtensor("int4 -> int8 fused, edge groups", g, (c, s_, z, None))

    for out_dt, tdt in ((qta.FP32, torch.float32), (qta.BF16, torch.bfloat16)):
        y = torch.empty((rows, cols), dtype=tdt, device=dev)
        qta.taco_decompress(d, dsh[0], y, out_dt)
        c0, s0b, z0b, _ = shards[0]
        ref = orc.decompress(orc.INT4_ASYM, 128, c0, s0b, z0b, None, 1, rows, cols,
                             orc.FP32 if out_dt == qta.FP32 else orc.BF16)
        torch.cuda.synchronize()
        assert_same(f"int4 decompress ({tdt}), edge groups", y, ref)
    assert qta.qta_device_error() == 0
