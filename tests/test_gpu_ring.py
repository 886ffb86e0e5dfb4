"""GPU parity of the ring hop (qar_dequant_add, qar_dequant_add_requant) and of
the ring reduce-scatter / all-reduce sequenced from it, against the oracle
on the same bytes: codes, scales, zeros, state and FP32 sums bit for bit."""
import numpy as np
import pytest
import torch

import oracle as orc
import quantized_tensor_activation_gb300 as qta
from quantized_tensor_activation_gb300 import ring
from gpu_util import (DT_TORCH, ORC_DT, ORC_SCH, assert_same, compare_qtensor, device, gpu_compress,
                      oracle_bits_in, oracle_compress, random_values, to_dtype_cpu)

pytestmark = pytest.mark.gpu

CASES = [(qta.TACO_FP8, 64), (qta.TACO_FP8, 128), (qta.TACO_FP8, 256), (qta.INT8_SYM_B64, 64),
         (qta.INT4_ASYM_G128, 128), (qta.INT8_ASYM_G128, 128)]
XDT = [qta.BF16, qta.FP16, qta.FP32]


def _incoming(scheme, B, batch, rows, cols, rng, dev):
    """A quantized partial sum, produced identically on both sides."""
    xt = to_dtype_cpu(random_values(rng, (batch, rows, cols), "mixed", 3.0), qta.FP32)
    d, q = gpu_compress(scheme, B, xt, qta.FP32, batch, rows, cols, qta.SCALE_CURRENT, dev=dev)
    ref = oracle_compress(scheme, B, xt, qta.FP32, batch, rows, cols, orc.CURRENT)
    compare_qtensor("incoming", q, ref)
    return d, q, ref


@pytest.mark.parametrize("scheme,B", CASES)
@pytest.mark.parametrize("xdt", XDT)
def test_dequant_add(scheme, B, xdt):
    dev = device()
    rng = np.random.default_rng(100 + 7 * scheme + B + xdt)
    batch, rows, cols = 2, 37, 1024          # 37 warp tiles, the last one ragged
    d, q, ref_in = _incoming(scheme, B, batch, rows, cols, rng, dev)
    xt = to_dtype_cpu(random_values(rng, (batch, rows, cols), "mixed"), xdt)
    out = torch.empty(batch * rows * cols, dtype=torch.float32, device=dev)
    qta.qar_dequant_add(d, q, xt.to(dev), xdt, out)
    ref = orc.dequant_add(ORC_SCH[scheme], B, *ref_in, batch, rows, cols, oracle_bits_in(xt), ORC_DT[xdt])
    assert_same("sum", out, ref)
    assert qta.qta_device_error() == 0


@pytest.mark.parametrize("scheme,B", CASES)
@pytest.mark.parametrize("xdt", XDT)
@pytest.mark.parametrize("mode", [qta.SCALE_DELAYED, qta.SCALE_CURRENT])
def test_dequant_add_requant(scheme, B, xdt, mode):
    if scheme != qta.TACO_FP8 and mode == qta.SCALE_DELAYED:
        pytest.skip("the scale mode only applies to TACO")
    dev = device()
    rng = np.random.default_rng(300 + 7 * scheme + B + xdt + 11 * mode)
    batch, rows, cols = 3, 21, 512
    d, q, ref_in = _incoming(scheme, B, batch, rows, cols, rng, dev)
    xt = to_dtype_cpu(random_values(rng, (batch, rows, cols), "mixed"), xdt)
    out = qta.alloc_qtensor(d, dev)
    st = None
    if scheme == qta.TACO_FP8:
        st = np.array([0.004, 0.0, 0.011, 0.0, 0.0007, 0.0], dtype=np.float32)   # S of the previous step
        out.state.copy_(torch.from_numpy(st))
    qta.qar_dequant_add_requant(d, q, xt.to(dev), xdt, out, mode)
    s = orc.dequant_add(ORC_SCH[scheme], B, *ref_in, batch, rows, cols, oracle_bits_in(xt), ORC_DT[xdt])
    c, sc, z = orc.compress(ORC_SCH[scheme], B, s, orc.FP32, batch, rows, cols, st, mode)
    compare_qtensor("requant", out, (c, sc, z, st))
    assert qta.qta_device_error() == 0


@pytest.mark.parametrize("scheme,B", [(qta.INT8_SYM_B64, 64), (qta.INT8_ASYM_G128, 128)])
def test_dequant_add_requant_many_tiles_per_warp(scheme, B):
    """The 8-warp INT8 hops on a call that spans the whole GPU: 8192 warp
    tiles, several per warp."""
    dev = device()
    rng = np.random.default_rng(900 + scheme)
    batch, rows, cols = 1, 8192, 2048
    d, q, ref_in = _incoming(scheme, B, batch, rows, cols, rng, dev)
    xt = to_dtype_cpu(random_values(rng, (batch, rows, cols), "mixed"), qta.BF16)
    out = qta.alloc_qtensor(d, dev)
    qta.qar_dequant_add_requant(d, q, xt.to(dev), qta.BF16, out, qta.SCALE_CURRENT)
    s = orc.dequant_add(ORC_SCH[scheme], B, *ref_in, batch, rows, cols, oracle_bits_in(xt), ORC_DT[qta.BF16])
    c, sc, z = orc.compress(ORC_SCH[scheme], B, s, orc.FP32, batch, rows, cols, None, qta.SCALE_CURRENT)
    compare_qtensor("requant", out, (c, sc, z, None))
    assert qta.qta_device_error() == 0


def _ring_inputs(n, rows, cols, dtype, seed):
    rng = np.random.default_rng(seed)
    return to_dtype_cpu(random_values(rng, (n, rows, cols), "mixed"), dtype)


@pytest.mark.parametrize("scheme,B", CASES)
@pytest.mark.parametrize("n,semi", [(2, False), (3, True), (4, False), (8, False), (8, True)])
def test_ring_allreduce_matches_oracle(scheme, B, n, semi):
    dev = device()
    rows, cols = 3 * n, 512
    xt = _ring_inputs(n, rows, cols, qta.BF16, 17 + n)
    s, y = ring.allreduce(qta.desc(scheme, B, rows, cols), xt.to(dev), semi, torch.float32)
    ref_s, ref_y = orc.ring_allreduce(ORC_SCH[scheme], B, [oracle_bits_in(xt[r]) for r in range(n)], orc.BF16,
                                      rows, cols, semi, orc.FP32)
    assert_same("reduce-scatter", s, ref_s)
    assert_same("all-reduce", y, ref_y)
    assert qta.qta_device_error() == 0


def test_ring_hop_partials_match_oracle_chains():
    dev = device()
    n, rows, cols = 4, 8, 1024
    xt = _ring_inputs(n, rows, cols, qta.FP16, 5)
    parts = []
    ring.reduce_scatter(qta.desc("int8_sym", 64, rows, cols), xt.to(dev), False, hop_partials=parts)
    rc = rows // n
    for j in range(n):
        order = [(j + k) % n for k in range(1, n)]
        for k in range(1, n):
            chunks = [oracle_bits_in(xt[r, j * rc:(j + 1) * rc].contiguous()) for r in order[:k]]
            q = orc.ring_chain(orc.INT8_SYM, 64, chunks, orc.FP16, rc, cols)
            ref = orc.decompress(orc.INT8_SYM, 64, *q, 1, rc, cols, orc.FP32)
            assert_same(f"chunk {j} after {k} ranks", parts[k - 1][j * rc:(j + 1) * rc], ref)


def test_ring_output_dtype_and_reuse():
    dev = device()
    n, rows, cols = 4, 16, 256
    xt = _ring_inputs(n, rows, cols, qta.BF16, 9).to(dev)
    d = qta.desc("taco_fp8", 128, rows, cols)
    a = ring.allreduce(d, xt, True, torch.bfloat16)
    b = ring.allreduce(d, xt, True, torch.bfloat16)      # every call starts afresh
    assert a[1].dtype == torch.bfloat16
    assert torch.equal(a[0], b[0]) and torch.equal(a[1].view(torch.int16), b[1].view(torch.int16))
    with pytest.raises(ValueError):
        ring.reduce_scatter(qta.desc("int8_sym", 64, 10, cols), xt[:, :10].contiguous())   # 10 % 4 != 0
