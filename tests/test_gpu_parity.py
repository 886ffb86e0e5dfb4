"""GPU parity: every kernel through the C ABI against the CPU oracle on the
same seeded inputs, element by element.  Codes, scales, zeros and per-tensor
state must be bit-exact; FP32 sums and decompressed values are expected
bit-exact and must be within max relative error 1e-5.

Shapes cover one block, one row, ragged tails (segment counts that are not a
multiple of the 32-segment warp tile), tensor boundaries inside a warp tile,
several tiles per warp (the stage ring wraps), every block size, every input
and output dtype, both scale modes, and 1..16 ranks."""
import numpy as np
import pytest
import torch

import oracle as orc
import quantized_tensor_activation_gb300 as qta
from gpu_util import (BLOCK_OF, ORC_DT, ORC_SCH, assert_close_f32, assert_same, compare_qtensor, device,
                      gpu_compress, oracle_bits_in, oracle_compress, random_values, to_dtype_cpu)

pytestmark = pytest.mark.gpu

DTYPES = [qta.BF16, qta.FP16, qta.FP32]
# (batch, rows, cols): one block, one row, ragged tiles with tensor boundaries
# inside warp tiles, many CTAs, and enough warp tiles to wrap the stage ring.
SHAPES = [(1, 1, 256), (3, 5, 512), (2, 37, 768), (4, 640, 1024), (4, 1024, 4096)]


@pytest.fixture(scope="module")
def dev():
    return device()


def _x(rng, batch, rows, cols, dtype, kind="mixed", scale=1.0):
    return to_dtype_cpu(random_values(rng, (batch, rows, cols), kind, scale), dtype)


@pytest.mark.parametrize("B", [64, 128, 256])
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", SHAPES)
def test_taco_compress_current(dev, B, dtype, shape):
    batch, rows, cols = shape
    rng = np.random.default_rng(hash((B, dtype, shape)) % 2 ** 32)
    xt = _x(rng, batch, rows, cols, dtype)
    _, q = gpu_compress(qta.TACO_FP8, B, xt, dtype, batch, rows, cols, qta.SCALE_CURRENT, dev=dev)
    ref = oracle_compress(qta.TACO_FP8, B, xt, dtype, batch, rows, cols, orc.CURRENT)
    torch.cuda.synchronize()
    compare_qtensor("taco", q, ref)


@pytest.mark.parametrize("B", [128, 256])
@pytest.mark.parametrize("dtype", [qta.BF16, qta.FP32])
def test_taco_compress_delayed_stale_scale(dev, B, dtype):
    # a previous-step scale far too small and one far too large: exercises
    # block-scale saturation (ratio > 448), codes saturating at 448, and the
    # r_b -> 2^-9 floor; amax accumulates onto the incoming value.
    batch, rows, cols = 3, 40, 1024
    rng = np.random.default_rng(B + dtype)
    xt = _x(rng, batch, rows, cols, dtype)
    state = np.array([1e-6, 0.5, 1e3, 0.0, 0.01, 7.0], dtype=np.float32)
    _, q = gpu_compress(qta.TACO_FP8, B, xt, dtype, batch, rows, cols, qta.SCALE_DELAYED, state=state, dev=dev)
    ref = oracle_compress(qta.TACO_FP8, B, xt, dtype, batch, rows, cols, orc.DELAYED, state=state)
    torch.cuda.synchronize()
    compare_qtensor("taco delayed", q, ref)
    assert (q.scales.cpu().numpy() == 0x7E).any()          # saturated block scales occurred


@pytest.mark.parametrize("scheme", [qta.INT8_SYM_B64, qta.INT4_ASYM_G128, qta.INT8_ASYM_G128])
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", SHAPES)
def test_int_compress(dev, scheme, dtype, shape):
    batch, rows, cols = shape
    B = BLOCK_OF[scheme]
    rng = np.random.default_rng(hash((scheme, dtype, shape)) % 2 ** 32)
    xt = _x(rng, batch, rows, cols, dtype, kind="t")
    _, q = gpu_compress(scheme, B, xt, dtype, batch, rows, cols, dev=dev)
    ref = oracle_compress(scheme, B, xt, dtype, batch, rows, cols)
    torch.cuda.synchronize()
    compare_qtensor(f"scheme {scheme}", q, ref)


def test_asym_fp32_extreme_range(dev):
    # fp32 sums beyond the fp16 range: the scale clamps at 65504 and the zero-
    # point at -65504; constant groups give s = 0.
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((2, 8, 512)) * 1e5).astype(np.float32)
    x[0, 3] = 2.5
    xt = torch.from_numpy(x)
    for scheme in (qta.INT4_ASYM_G128, qta.INT8_ASYM_G128):
        _, q = gpu_compress(scheme, 128, xt, qta.FP32, 2, 8, 512, dev=dev)
        ref = oracle_compress(scheme, 128, xt, qta.FP32, 2, 8, 512)
        torch.cuda.synchronize()
        compare_qtensor("asym extreme", q, ref)


def test_zero_and_constant_tensors(dev):
    for scheme, B in ((qta.TACO_FP8, 128), (qta.INT8_SYM_B64, 64), (qta.INT4_ASYM_G128, 128)):
        for val in (0.0, -3.0):
            xt = torch.full((2, 3, 256), val, dtype=torch.bfloat16)
            _, q = gpu_compress(scheme, B, xt, qta.BF16, 2, 3, 256, dev=dev)
            ref = oracle_compress(scheme, B, xt, qta.BF16, 2, 3, 256)
            torch.cuda.synchronize()
            compare_qtensor(f"const {val}", q, ref)


def _tie_blocks(rng, n_blocks, B):
    """Blocks whose butterflies meet exact zeros of every sign: upper half a
    copy of the lower half (the last stage subtracts equal values), every
    stride-64 partner equal, blocks of random +0 / -0, and the rest mixed
    values with signed zeros sprinkled in."""
    x = random_values(rng, (n_blocks, B), "mixed")
    kind = rng.integers(0, 4, n_blocks)
    h = B // 2
    x[kind == 1, h:] = x[kind == 1, :h]
    if B >= 128:
        for lo in range(0, B, 128):
            x[kind == 2, lo + 64:lo + 128] = x[kind == 2, lo:lo + 64]
    zeros = np.where(rng.random((n_blocks, B)) < 0.5, np.float32(-0.0), np.float32(0.0))
    x[kind == 3] = zeros[kind == 3]
    sprinkle = rng.random((n_blocks, B)) < 0.1
    x[sprinkle & (kind == 0)[:, None]] = zeros[sprinkle & (kind == 0)[:, None]]
    return x


@pytest.mark.parametrize("B", [64, 128, 256])
@pytest.mark.parametrize("dtype", DTYPES)
def test_taco_compress_signed_zeros_and_ties(dev, B, dtype):
    # the cross-lane stages form (lower - upper) in whichever lane keeps the
    # position; equal operands and signed zeros must give the oracle's zero
    # signs, hence its codes (0x00 vs 0x80), bit for bit
    batch, rows, cols = 3, 21, 1024
    rng = np.random.default_rng(7 * B + dtype)
    x = _tie_blocks(rng, batch * rows * cols // B, B).reshape(batch, rows, cols)
    xt = to_dtype_cpu(x, dtype)
    for mode in (qta.SCALE_CURRENT, qta.SCALE_DELAYED):
        state = np.array([0.002, 0.0, 0.0, 0.0, 1e-5, 0.0], dtype=np.float32)
        _, q = gpu_compress(qta.TACO_FP8, B, xt, dtype, batch, rows, cols, mode, state=state.copy(), dev=dev)
        ref = oracle_compress(qta.TACO_FP8, B, xt, dtype, batch, rows, cols,
                              orc.CURRENT if mode == qta.SCALE_CURRENT else orc.DELAYED, state=state.copy())
        torch.cuda.synchronize()
        compare_qtensor(f"ties mode {mode}", q, ref)


@pytest.mark.parametrize("B", [64, 128, 256])
@pytest.mark.parametrize("out_dtype", DTYPES)
def test_taco_decompress_signed_zeros_and_ties(dev, B, out_dtype):
    # codes drawn from few values with many +-0 (0x00 / 0x80) and with halves
    # and stride-64 partners repeated, so the inverse butterflies meet equal
    # operands and signed zeros
    batch, rows, cols = 2, 19, 1024
    n = batch * rows * cols
    rng = np.random.default_rng(11 * B + out_dtype)
    pool = np.array([0x00, 0x80, 0x00, 0x80, 0x38, 0xB8, 0x01, 0x81, 0x7E, 0xFE], dtype=np.uint8)
    c = pool[rng.integers(0, pool.size, n)].reshape(-1, B)
    kind = rng.integers(0, 3, c.shape[0])
    c[kind == 1, B // 2:] = c[kind == 1, :B // 2]
    if B >= 128:
        for lo in range(0, B, 128):
            c[kind == 2, lo + 64:lo + 128] = c[kind == 2, lo:lo + 64]
    c = c.reshape(-1)
    s = rng.integers(0x08, 0x7E, n // B).astype(np.uint8)
    st = np.array([0.003, 0.0, 1.5, 0.0], dtype=np.float32)
    d = qta.desc(qta.TACO_FP8, B, rows, cols, batch=batch)
    q = qta.QTensor(d, torch.from_numpy(c).to(dev), torch.from_numpy(s).to(dev), None, torch.from_numpy(st).to(dev))
    y = torch.empty((batch, rows, cols), dtype={0: torch.bfloat16, 1: torch.float16, 2: torch.float32}[out_dtype],
                    device=dev)
    qta.taco_decompress(d, q, y, out_dtype)
    ref = orc.decompress(orc.TACO_FP8, B, c, s, None, st, batch, rows, cols, ORC_DT[out_dtype])
    torch.cuda.synchronize()
    assert_same("decompress ties", y, ref)


@pytest.mark.parametrize("scheme,B", [(qta.TACO_FP8, 64), (qta.TACO_FP8, 128), (qta.TACO_FP8, 256),
                                      (qta.INT8_SYM_B64, 64), (qta.INT4_ASYM_G128, 128),
                                      (qta.INT8_ASYM_G128, 128)])
@pytest.mark.parametrize("out_dtype", DTYPES)
@pytest.mark.parametrize("shape", [(1, 1, 256), (3, 5, 512), (4, 640, 1024), (2, 2048, 4096)])
def test_decompress(dev, scheme, B, out_dtype, shape):
    batch, rows, cols = shape
    rng = np.random.default_rng(hash((scheme, B, out_dtype, shape)) % 2 ** 32)
    xt = _x(rng, batch, rows, cols, qta.FP32, kind="mixed")
    # the oracle's codes are the decompressor's input on both sides
    c, s, z, st = oracle_compress(scheme, B, xt, qta.FP32, batch, rows, cols)
    d = qta.desc(scheme, B, rows, cols, batch=batch)
    q = qta.QTensor(d, torch.from_numpy(c.view(np.uint8)).to(dev), torch.from_numpy(s.view(np.uint8)).to(dev),
                    None if z is None else torch.from_numpy(z.view(np.uint8)).to(dev),
                    None if st is None else torch.from_numpy(st).to(dev))
    y = torch.empty((batch, rows, cols), dtype={0: torch.bfloat16, 1: torch.float16, 2: torch.float32}[out_dtype],
                    device=dev)
    qta.taco_decompress(d, q, y, out_dtype)
    ref = orc.decompress(ORC_SCH[scheme], B, c, s, z, st, batch, rows, cols, ORC_DT[out_dtype])
    torch.cuda.synchronize()
    assert_same("decompress", y, ref)
    if out_dtype == qta.FP32:
        assert_close_f32("decompress fp32", y, ref)


def _oracle_shards(scheme, B, n, rows, cols, rng, dtype=qta.BF16):
    shards, dev_shards = [], []
    for r in range(n):
        xt = to_dtype_cpu(random_values(rng, (rows, cols), "mixed", scale=1.0 + r), dtype)
        c, s, z, st = oracle_compress(scheme, B, xt, dtype, 1, rows, cols)
        shards.append((c, s, z, st))
    return shards


def _to_dev(scheme, B, rows, cols, shards, dev):
    d = qta.desc(scheme, B, rows, cols)
    out = []
    for c, s, z, st in shards:
        out.append(qta.QTensor(d, torch.from_numpy(c.view(np.uint8).copy()).to(dev),
                               torch.from_numpy(s.view(np.uint8).copy()).to(dev),
                               None if z is None else torch.from_numpy(z.view(np.uint8).copy()).to(dev),
                               None if st is None else torch.from_numpy(st.copy()).to(dev)))
    return d, out


@pytest.mark.parametrize("scheme,B", [(qta.TACO_FP8, 64), (qta.TACO_FP8, 128), (qta.TACO_FP8, 256),
                                      (qta.INT8_SYM_B64, 64), (qta.INT4_ASYM_G128, 128),
                                      (qta.INT8_ASYM_G128, 128)])
@pytest.mark.parametrize("n", [1, 2, 3, 4, 8, 16])
def test_reduce(dev, scheme, B, n):
    rows, cols = 96, 1024
    rng = np.random.default_rng(hash((scheme, B, n)) % 2 ** 32)
    shards = _oracle_shards(scheme, B, n, rows, cols, rng)
    d, ds = _to_dev(scheme, B, rows, cols, shards, dev)
    for rb, re_ in ((0, rows), (7, 61), (95, 96)):
        out = torch.full((re_ - rb, cols), float("nan"), dtype=torch.float32, device=dev)
        qta.qar_reduce(d, ds, rb, re_, out)
        ref = orc.reduce(ORC_SCH[scheme], B, shards, rows, cols, rb, re_)
        torch.cuda.synchronize()
        assert_same(f"reduce rows {rb}:{re_}", out, ref)
        assert_close_f32("reduce", out, ref)


def test_reduce_many_tiles(dev):
    # enough output segments that every warp of the persistent grid loops over
    # several tiles and its (tile, rank) stage ring wraps many times
    scheme, B, n, rows, cols = qta.TACO_FP8, 128, 8, 2048, 4096
    rng = np.random.default_rng(11)
    shards = _oracle_shards(scheme, B, n, rows, cols, rng)
    d, ds = _to_dev(scheme, B, rows, cols, shards, dev)
    out = torch.empty((rows, cols), dtype=torch.float32, device=dev)
    qta.qar_reduce(d, ds, 0, rows, out)
    ref = orc.reduce(orc.TACO_FP8, B, shards, rows, cols)
    torch.cuda.synchronize()
    assert_same("reduce many tiles", out, ref)


@pytest.mark.parametrize("n", [4, 8])
def test_reduce_int4_many_tiles(dev, n):
    # the INT4 reduces compiled for 4 and 8 shards issue each TMA load from
    # the unit's constant position STAGES units ahead: with the grid capped to
    # 2 SMs every warp runs about 32 tiles, so that position crosses tiles
    rows, cols = 1024, 2048
    rng = np.random.default_rng(17 + n)
    shards = _oracle_shards(qta.INT4_ASYM_G128, 128, n, rows, cols, rng, dtype=qta.FP16)
    d, ds = _to_dev(qta.INT4_ASYM_G128, 128, rows, cols, shards, dev)
    d.max_sms = 2
    out = torch.empty((rows, cols), dtype=torch.float32, device=dev)
    qta.qar_reduce(d, ds, 0, rows, out)
    ref = orc.reduce(orc.INT4_ASYM, 128, shards, rows, cols)
    torch.cuda.synchronize()
    assert_same(f"int4 reduce, {n} shards, many tiles", out, ref)
    nb = 4
    dg = qta.desc(qta.INT8_ASYM_G128, 128, rows // nb, cols, batch=nb)
    g = qta.alloc_qtensor(dg, dev)
    qta.qar_reduce_requant(d, ds, 0, rows, dg, g, qta.SCALE_CURRENT)
    c, s_, z = orc.reduce_requant(orc.INT4_ASYM, 128, shards, rows, cols, 0, rows, orc.INT8_ASYM, 128, nb, None,
                                  orc.CURRENT)
    torch.cuda.synchronize()
    compare_qtensor(f"int4 -> int8 fused, {n} shards, many tiles", g, (c, s_, z, None))
    assert qta.qta_device_error() == 0


@pytest.mark.parametrize("n", [4, 8])
def test_reduce_int4_row_ranges(dev, n):
    # 10 segments per row and 63 rows, reduced over rows 0:63, 16:48 and 3:50
    # by the 4- and 8-shard INT4 reduces: tiles that start mid-row, a first
    # segment that is not a multiple of 32 (rows 3:50 start at segment 30),
    # and a last warp tile of 0:63 that reaches past the end of the arrays
    # (its rows are read as zeros and its lanes store nothing)
    rows, cols = 63, 640
    rng = np.random.default_rng(23 + n)
    shards = _oracle_shards(qta.INT4_ASYM_G128, 128, n, rows, cols, rng, dtype=qta.FP16)
    d, ds = _to_dev(qta.INT4_ASYM_G128, 128, rows, cols, shards, dev)
    for rb, re_ in ((0, rows), (16, 48), (3, 50)):
        out = torch.empty((re_ - rb, cols), dtype=torch.float32, device=dev)
        qta.qar_reduce(d, ds, rb, re_, out)
        ref = orc.reduce(orc.INT4_ASYM, 128, shards, rows, cols, rb, re_)
        torch.cuda.synchronize()
        assert_same(f"int4 reduce rows {rb}:{re_}, {n} shards", out, ref)
        nb = 1
        dg = qta.desc(qta.INT8_ASYM_G128, 128, re_ - rb, cols, batch=nb)
        g = qta.alloc_qtensor(dg, dev)
        qta.qar_reduce_requant(d, ds, rb, re_, dg, g, qta.SCALE_CURRENT)
        c, s_, z = orc.reduce_requant(orc.INT4_ASYM, 128, shards, rows, cols, rb, re_, orc.INT8_ASYM, 128, nb, None,
                                      orc.CURRENT)
        torch.cuda.synchronize()
        compare_qtensor(f"int4 -> int8 fused rows {rb}:{re_}, {n} shards", g, (c, s_, z, None))
    assert qta.qta_device_error() == 0


def test_taco_steps_with_drift(dev):
    # successive steps with a per-step magnitude drift: step 0 CURRENT, later
    # steps DELAYED with the scale left by taco_update_scale of the previous
    # step, on both sides.
    batch, rows, cols, B = 2, 64, 1024, 256
    rng = np.random.default_rng(3)
    base = random_values(rng, (batch, rows, cols), "normal", 1e-4)
    d = qta.desc(qta.TACO_FP8, B, rows, cols, batch=batch)
    q = qta.alloc_qtensor(d, dev)
    st = np.zeros(2 * batch, dtype=np.float32)
    for step in range(8):
        f = float(np.exp(rng.uniform(np.log(0.25), np.log(4.0))))
        xt = to_dtype_cpu((base * np.float32(f)).astype(np.float32), qta.BF16)
        mode = qta.SCALE_CURRENT if step == 0 else qta.SCALE_DELAYED
        qta.taco_compress(d, xt.to(dev), qta.BF16, q, mode)
        c, s, _ = orc.compress(orc.TACO_FP8, B, oracle_bits_in(xt), orc.BF16, batch, rows, cols, st,
                               orc.CURRENT if step == 0 else orc.DELAYED)
        torch.cuda.synchronize()
        assert_same(f"step {step} codes", q.codes, c)
        assert_same(f"step {step} scales", q.scales, s)
        assert_same(f"step {step} state", q.state, st)
        qta.taco_update_scale(q.state, batch)
        orc.taco_update_scale(st)
        torch.cuda.synchronize()
        assert_same(f"step {step} updated state", q.state, st)


def test_requant_full_chain(dev):
    # compress -> reduce -> requant -> decompress for each workload's scheme
    # pair, at a reduced size, bit-exact at every stage
    cases = [(qta.TACO_FP8, 128, qta.TACO_FP8, 128, qta.BF16, 4),
             (qta.INT8_SYM_B64, 64, qta.INT8_SYM_B64, 64, qta.BF16, 8),
             (qta.INT4_ASYM_G128, 128, qta.INT8_ASYM_G128, 128, qta.FP16, 8)]
    for sch, B, gsch, gB, dtype, N in cases:
        R, C = 128, 1024
        rng = np.random.default_rng(sch)
        xt = to_dtype_cpu(random_values(rng, (N, R, C), "t"), dtype)
        d, q = gpu_compress(sch, B, xt, dtype, N, R, C, dev=dev)
        ref = oracle_compress(sch, B, xt, dtype, N, R, C)
        d1 = qta.desc(sch, B, R, C)
        ssum = torch.empty((R, C), dtype=torch.float32, device=dev)
        qta.qar_reduce(d1, [q.shard(r) for r in range(N)], 0, R, ssum)
        E = R * C
        nb = E // B
        cb = E // 2 if sch == qta.INT4_ASYM_G128 else E
        shards = [(ref[0][r * cb:(r + 1) * cb], ref[1][r * nb:(r + 1) * nb],
                   None if ref[2] is None else ref[2][r * nb:(r + 1) * nb],
                   None if ref[3] is None else ref[3][2 * r:2 * r + 2]) for r in range(N)]
        osum = orc.reduce(ORC_SCH[sch], B, shards, R, C)
        dg = qta.desc(gsch, gB, R // N, C, batch=N)
        g = qta.alloc_qtensor(dg, dev)
        qta.qar_requant(dg, ssum, g, qta.SCALE_CURRENT)
        gref = oracle_compress(gsch, gB, torch.from_numpy(osum.reshape(R, C)), qta.FP32, N, R // N, C)
        y = torch.empty((R, C), dtype=torch.bfloat16 if dtype == qta.BF16 else torch.float16, device=dev)
        qta.taco_decompress(dg, g, y, dtype)
        yref = orc.decompress(ORC_SCH[gsch], gB, *gref, N, R // N, C, ORC_DT[dtype])
        torch.cuda.synchronize()
        compare_qtensor("stage-1", q, ref)
        assert_same("sum", ssum, osum)
        compare_qtensor("requant", g, gref)
        assert_same("output", y, yref)


def test_error_status_leaves_outputs_untouched(dev):
    d = qta.desc(qta.TACO_FP8, 128, 4, 256)
    q = qta.alloc_qtensor(d, dev)
    q.codes.fill_(0xA5)
    x = torch.randn(4 * 256 + 8, dtype=torch.bfloat16, device=dev)
    with pytest.raises(qta.QtaError) as e:
        qta.taco_compress(d, x.data_ptr() + 2, qta.BF16, q)      # misaligned input
    assert e.value.status == qta.QTA_ERR_ALIGNMENT
    with pytest.raises(qta.QtaError) as e:
        qta.qar_reduce(d, [q.shard(0)] * 17, 0, 4, torch.empty(4, 256, device=dev))
    assert e.value.status == qta.QTA_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert (q.codes == 0xA5).all()
    assert qta.qta_device_error() == 0


def test_copy_kernel(dev):
    n = (1 << 24) + 48
    src = torch.randint(0, 255, (n,), dtype=torch.uint8, device=dev)
    dst = torch.zeros_like(src)
    qta.qta_copy(src, dst, n)
    torch.cuda.synchronize()
    assert torch.equal(src, dst)


@pytest.mark.parametrize("scheme,B,gscheme,gB", [(qta.TACO_FP8, 128, qta.TACO_FP8, 128),
                                                 (qta.TACO_FP8, 256, qta.TACO_FP8, 256),
                                                 (qta.TACO_FP8, 256, qta.TACO_FP8, 128),
                                                 (qta.TACO_FP8, 64, qta.TACO_FP8, 256),
                                                 (qta.INT8_SYM_B64, 64, qta.INT8_SYM_B64, 64),
                                                 (qta.INT4_ASYM_G128, 128, qta.INT8_ASYM_G128, 128),
                                                 (qta.INT8_ASYM_G128, 128, qta.INT8_ASYM_G128, 128)])
@pytest.mark.parametrize("n", [1, 3, 4, 8])
@pytest.mark.parametrize("mode", [qta.SCALE_CURRENT, qta.SCALE_DELAYED])
def test_reduce_requant_fused(dev, scheme, B, gscheme, gB, n, mode):
    # the fused call against the oracle's fused reduce + requant (TACO ->
    # TACO with equal blocks requantizes the Hadamard-domain sums; every
    # other pair is reduce, then compress of the FP32 sum), bit for bit
    rows, cols = 96, 1024
    rng = np.random.default_rng(hash((scheme, B, gscheme, n, mode)) % 2 ** 32)
    shards = _oracle_shards(scheme, B, n, rows, cols, rng)
    d, ds = _to_dev(scheme, B, rows, cols, shards, dev)
    for rb, re_, nb in ((0, rows, 4), (8, 56, 3), (95, 96, 1)):
        gr = (re_ - rb) // nb
        dg = qta.desc(gscheme, gB, gr, cols, batch=nb)
        g = qta.alloc_qtensor(dg, dev)
        st0 = None
        if g.state is not None:
            st0 = np.zeros(2 * nb, dtype=np.float32)
            st0[0::2] = [0.003 * (j + 1) for j in range(nb)]
            st0[1::2] = [0.5 * j for j in range(nb)]
            g.state.copy_(torch.from_numpy(st0))
        qta.qar_reduce_requant(d, ds, rb, re_, dg, g, mode)
        st_ref = None if st0 is None else st0.copy()
        c, s, z = orc.reduce_requant(ORC_SCH[scheme], B, shards, rows, cols, rb, re_, ORC_SCH[gscheme], gB,
                                     nb, st_ref, orc.CURRENT if mode == qta.SCALE_CURRENT else orc.DELAYED)
        ref = (c, s, z, st_ref)
        torch.cuda.synchronize()
        compare_qtensor(f"fused rows {rb}:{re_}", g, ref)
    assert qta.qta_device_error() == 0


def test_reduce_requant_rejects_unsupported_pairs(dev):
    d = qta.desc(qta.TACO_FP8, 128, 8, 256)
    q = qta.alloc_qtensor(d, dev)
    dg = qta.desc(qta.INT8_SYM_B64, 64, 8, 256)
    g = qta.alloc_qtensor(dg, dev)
    with pytest.raises(qta.QtaError) as e:
        qta.qar_reduce_requant(d, [q], 0, 8, dg, g)
    assert e.value.status == qta.QTA_ERR_UNSUPPORTED
    with pytest.raises(qta.QtaError) as e:
        qta.qar_reduce_requant(d, [q], 0, 8, qta.desc(qta.TACO_FP8, 128, 3, 256, batch=2), q)
    assert e.value.status == qta.QTA_ERR_INVALID_ARG


@pytest.mark.parametrize("B", [64, 128, 256])
@pytest.mark.parametrize("dtype", [qta.BF16, qta.FP32])
@pytest.mark.parametrize("mode", [qta.SCALE_CURRENT, qta.SCALE_DELAYED])
def test_taco_compress_round_up(dev, B, dtype, mode):
    # block scales rounded up to the smallest covering E4M3 value, with the
    # same stale previous-step scales as above in DELAYED mode
    batch, rows, cols = 3, 37, 1024
    rng = np.random.default_rng(7 * B + dtype + 3 * mode)
    xt = _x(rng, batch, rows, cols, dtype)
    state = np.array([1e-6, 0.5, 1e3, 0.0, 0.01, 7.0], dtype=np.float32)
    _, q = gpu_compress(qta.TACO_FP8, B, xt, dtype, batch, rows, cols, mode | qta.SCALE_ROUND_UP, state=state,
                        dev=dev)
    omode = (orc.CURRENT if mode == qta.SCALE_CURRENT else orc.DELAYED) | orc.ROUND_UP
    ref = oracle_compress(qta.TACO_FP8, B, xt, dtype, batch, rows, cols, omode, state=state)
    torch.cuda.synchronize()
    compare_qtensor("taco round-up", q, ref)


@pytest.mark.parametrize("gB", [128, 256])
def test_reduce_requant_round_up(dev, gB):
    rows, cols, n, nb = 64, 1024, 4, 4
    rng = np.random.default_rng(gB)
    shards = _oracle_shards(qta.TACO_FP8, 128, n, rows, cols, rng)
    d, ds = _to_dev(qta.TACO_FP8, 128, rows, cols, shards, dev)
    dg = qta.desc(qta.TACO_FP8, gB, rows // nb, cols, batch=nb)
    g = qta.alloc_qtensor(dg, dev)
    qta.qar_reduce_requant(d, ds, 0, rows, dg, g, qta.SCALE_CURRENT | qta.SCALE_ROUND_UP)
    st_ref = np.zeros(2 * nb, dtype=np.float32)
    c, s, z = orc.reduce_requant(orc.TACO_FP8, 128, shards, rows, cols, 0, rows, orc.TACO_FP8, gB, nb, st_ref,
                                 orc.CURRENT | orc.ROUND_UP)
    torch.cuda.synchronize()
    compare_qtensor("fused round-up", g, (c, s, z, st_ref))
    assert qta.qta_device_error() == 0
