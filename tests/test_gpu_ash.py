"""GPU parity of the adaptive rescaling (the per-channel powers of two of
TACO's Adaptive Scale-Hadamard transform; TACO Core claim, Fig. 7) against
the oracle, bit for bit: the per-channel amax, the factor update, and the
compress, decompress, FP32 reduce, fused reduce + requant and requant with
the factors."""
import numpy as np
import pytest
import torch

import oracle as orc
import quantized_tensor_activation_gb300 as qta
from gpu_util import ORC_DT, assert_same, bits, device, oracle_bits_in, random_values, to_dtype_cpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return device()


def _outlier_x(rng, shape, dtype, n_out=None):
    x = random_values(rng, shape, "laplace")
    cols = shape[-1]
    ch = rng.choice(cols, n_out or max(1, cols // 50), replace=False)
    x[..., ch] *= rng.uniform(8, 200, size=len(ch)).astype(np.float32)
    return to_dtype_cpu(x, dtype)


def _chan_for(xt, dtype, batch, rows, cols, dev):
    """Factors from the data itself, on both sides (GPU and oracle)."""
    c = qta.alloc_chan(cols, dev)
    d = qta.desc(qta.TACO_FP8, 64, rows, cols, batch=batch)
    qta.taco_channel_amax(d, xt.to(dev), dtype, c)
    qta.taco_ash_update(c, cols)
    oc = orc.new_chan_state(cols)
    orc.channel_amax(oracle_bits_in(xt), ORC_DT[dtype], batch, rows, cols, oc)
    orc.ash_update(oc, cols)
    torch.cuda.synchronize()
    assert_same("channel factors", c, oc)
    return c, oc


@pytest.mark.parametrize("dtype", [qta.BF16, qta.FP16, qta.FP32])
@pytest.mark.parametrize("shape", [(1, 1, 64), (2, 37, 192), (3, 300, 1024)])
def test_channel_amax(dev, dtype, shape):
    batch, rows, cols = shape
    rng = np.random.default_rng(rows + cols + dtype)
    xt = _outlier_x(rng, shape, dtype)
    c = qta.alloc_chan(cols, dev)
    c[2 * cols::7] = 0.75                                   # max-accumulates onto earlier values
    oc = orc.new_chan_state(cols)
    oc[2 * cols::7] = 0.75
    qta.taco_channel_amax(qta.desc(qta.TACO_FP8, 64, rows, cols, batch=batch), xt.to(dev), dtype, c)
    orc.channel_amax(oracle_bits_in(xt), ORC_DT[dtype], batch, rows, cols, oc)
    torch.cuda.synchronize()
    assert_same("channel amax", c, oc)
    assert qta.qta_device_error() == 0


@pytest.mark.parametrize("cols", [64, 1000, 8192, 65536])
def test_ash_update(dev, cols):
    rng = np.random.default_rng(cols)
    am = (np.exp(rng.uniform(-40, 30, cols)) * (rng.random(cols) < 0.9)).astype(np.float32)
    am[: cols // 3] = np.float32(0.01) * np.exp2(rng.integers(-2, 8, cols // 3)).astype(np.float32)
    if cols >= 1000:
        am[5] = np.float32(1e-42)                             # subnormal
        am[6] = 0.0
    oc = orc.new_chan_state(cols)
    oc[2 * cols:] = am
    c = torch.from_numpy(oc.copy()).to(dev)
    qta.taco_ash_update(c, cols)
    orc.ash_update(oc, cols)
    torch.cuda.synchronize()
    assert_same("ash update", c, oc)


@pytest.mark.parametrize("B", [64, 128, 256])
@pytest.mark.parametrize("dtype", [qta.BF16, qta.FP32])
@pytest.mark.parametrize("mode", [qta.SCALE_CURRENT, qta.SCALE_DELAYED])
def test_compress_decompress_with_factors(dev, B, dtype, mode):
    batch, rows, cols = 3, 37, 1024
    rng = np.random.default_rng(B + 10 * dtype + mode)
    xt = _outlier_x(rng, (batch, rows, cols), dtype)
    c, oc = _chan_for(xt, dtype, batch, rows, cols, dev)
    assert (oc[:cols] < 1).any()
    d = qta.desc(qta.TACO_FP8, B, rows, cols, batch=batch)
    q = qta.alloc_qtensor(d, dev)
    q.chan = c
    st = np.zeros(2 * batch, np.float32)
    st[0::2] = [0.02, 0.5, 0.001]
    q.state.copy_(torch.from_numpy(st))
    qta.taco_compress(d, xt.to(dev), dtype, q, mode)
    oco, osc, _ = orc.compress(orc.TACO_FP8, B, oracle_bits_in(xt), ORC_DT[dtype], batch, rows, cols, st,
                               orc.CURRENT if mode == qta.SCALE_CURRENT else orc.DELAYED, chan=oc)
    torch.cuda.synchronize()
    assert_same("codes", q.codes, oco)
    assert_same("scales", q.scales, osc)
    assert_same("state", q.state, st)
    for od in (qta.BF16, qta.FP16, qta.FP32):
        y = torch.empty((batch, rows, cols), dtype={qta.BF16: torch.bfloat16, qta.FP16: torch.float16,
                                                    qta.FP32: torch.float32}[od], device=dev)
        qta.taco_decompress(d, q, y, od)
        yo = orc.decompress(orc.TACO_FP8, B, oco, osc, None, st, batch, rows, cols, ORC_DT[od], chan=oc)
        torch.cuda.synchronize()
        assert_same(f"decompress {od}", y, yo)
    assert qta.qta_device_error() == 0


@pytest.mark.parametrize("B,gB", [(128, 128), (256, 256), (128, 256), (256, 64)])
@pytest.mark.parametrize("n", [1, 3, 8])
def test_reduce_and_fused_with_factors(dev, B, gB, n):
    rows, cols = 64, 2048
    rng = np.random.default_rng(B + gB + n)
    xt = _outlier_x(rng, (n, rows, cols), qta.BF16)
    c, oc = _chan_for(xt, qta.BF16, n, rows, cols, dev)
    d = qta.desc(qta.TACO_FP8, B, rows, cols, batch=n)
    q = qta.alloc_qtensor(d, dev)
    q.chan = c
    qta.taco_compress(d, xt.to(dev), qta.BF16, q, qta.SCALE_CURRENT)
    st = np.zeros(2 * n, np.float32)
    oco, osc, _ = orc.compress(orc.TACO_FP8, B, oracle_bits_in(xt), orc.BF16, n, rows, cols, st, orc.CURRENT,
                               chan=oc)
    E, nb = rows * cols, rows * cols // B
    shards = [(oco[r * E:(r + 1) * E], osc[r * nb:(r + 1) * nb], None, st[2 * r:2 * r + 2]) for r in range(n)]
    d1 = qta.desc(qta.TACO_FP8, B, rows, cols)
    sh = [q.shard(r) for r in range(n)]
    s = torch.empty((rows - 8, cols), dtype=torch.float32, device=dev)
    qta.qar_reduce(d1, sh, 8, rows, s)
    so = orc.reduce(orc.TACO_FP8, B, shards, rows, cols, 8, rows, chan=oc)
    torch.cuda.synchronize()
    assert_same("reduce sum", s, so)
    nb_out = 4
    dg = qta.desc(qta.TACO_FP8, gB, rows // nb_out, cols, batch=nb_out)
    g = qta.alloc_qtensor(dg, dev)
    g.chan = c
    gst = np.zeros(2 * nb_out, np.float32)
    gst[0::2] = 0.05
    g.state.copy_(torch.from_numpy(gst))
    qta.qar_reduce_requant(d1, sh, 0, rows, dg, g, qta.SCALE_DELAYED)
    gc, gs, _ = orc.reduce_requant(orc.TACO_FP8, B, shards, rows, cols, 0, rows, orc.TACO_FP8, gB, nb_out, gst,
                                   orc.DELAYED, chan=oc)
    torch.cuda.synchronize()
    assert_same("fused codes", g.codes, gc)
    assert_same("fused scales", g.scales, gs)
    assert_same("fused state", g.state, gst)
    # the requant of an FP32 sum with the factors
    s2 = torch.empty((rows, cols), dtype=torch.float32, device=dev)
    qta.qar_reduce(d1, sh, 0, rows, s2)
    g2 = qta.alloc_qtensor(dg, dev)
    g2.chan = c
    qta.qar_requant(dg, s2, g2, qta.SCALE_CURRENT)
    st3 = np.zeros(2 * nb_out, np.float32)
    so2 = orc.reduce(orc.TACO_FP8, B, shards, rows, cols, chan=oc)
    rc, rs, _ = orc.compress(orc.TACO_FP8, gB, so2, orc.FP32, nb_out, rows // nb_out, cols, st3, orc.CURRENT,
                             chan=oc)
    torch.cuda.synchronize()
    assert_same("requant codes", g2.codes, rc)
    assert_same("requant scales", g2.scales, rs)
    assert_same("requant state", g2.state, st3)
    assert qta.qta_device_error() == 0


def test_rescaling_lowers_the_round_trip_error(dev):
    # outlier channels (the Flash-style workload's kind): the rescaled round
    # trip is closer to the input than the plain one
    import workloads
    w = workloads.WORKLOADS["flash_int4"]
    x = workloads.make_rank_inputs(w, rows=512, ranks=1, device=dev)[0]
    R, C = x.shape
    d = qta.desc(qta.TACO_FP8, 128, R, C)
    c = qta.alloc_chan(C, dev)
    qta.taco_channel_amax(d, x, qta.FP16, c)
    qta.taco_ash_update(c, C)
    errs = []
    for chan in (None, c):
        q = qta.alloc_qtensor(d, dev)
        q.chan = chan
        qta.taco_compress(d, x, qta.FP16, q, qta.SCALE_CURRENT)
        y = torch.empty((R, C), dtype=torch.float32, device=dev)
        qta.taco_decompress(d, q, y, qta.FP32)
        errs.append(float(((y.double() - x.double()) ** 2).mean()))
    assert errs[1] < 0.6 * errs[0], errs


def test_factor_argument_checks(dev):
    rows, cols = 8, 256
    d = qta.desc(qta.TACO_FP8, 128, rows, cols, batch=2)
    q = qta.alloc_qtensor(d, dev)
    c1, c2 = qta.alloc_chan(cols, dev), qta.alloc_chan(cols, dev)
    q.chan = c1
    x = torch.zeros((2, rows, cols), dtype=torch.bfloat16, device=dev)
    qta.taco_compress(d, x, qta.BF16, q)
    sh = [q.shard(0), q.shard(1)]
    sh[1].chan = c2
    d1 = qta.desc(qta.TACO_FP8, 128, rows, cols)
    with pytest.raises(qta.QtaError) as e:
        qta.qar_reduce(d1, sh, 0, rows, torch.empty((rows, cols), device=dev))
    assert e.value.status == qta.QTA_ERR_INVALID_ARG                  # ranks with different factors
    sh[1].chan = c1
    g = qta.alloc_qtensor(qta.desc(qta.TACO_FP8, 128, rows // 2, cols, batch=2), dev)
    g.chan = c2
    with pytest.raises(qta.QtaError) as e:
        qta.qar_reduce_requant(d1, sh, 0, rows, g.desc, g)
    assert e.value.status == qta.QTA_ERR_UNSUPPORTED                  # other factors on the output
    qi = qta.alloc_qtensor(qta.desc(qta.INT8_SYM_B64, 64, rows, cols), dev)
    qi.chan = c1
    with pytest.raises(qta.QtaError) as e:
        qta.taco_compress(qi.desc, x[0], qta.BF16, qi)
    assert e.value.status == qta.QTA_ERR_UNSUPPORTED                  # factors go with TACO only
    out = qta.alloc_qtensor(d1, dev)
    with pytest.raises(qta.QtaError) as e:
        qta.qar_dequant_add_requant(d1, sh[0], x[1], qta.BF16, out)
    assert e.value.status == qta.QTA_ERR_UNSUPPORTED                  # no rescaling in the ring hops
    torch.cuda.synchronize()
    assert qta.qta_device_error() == 0
