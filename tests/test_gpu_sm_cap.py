"""Capping the SMs a call occupies (qta_desc.max_sms) changes the persistent
grid only: every call gives the same bytes with 1, 7 or all SMs, which also
walks each warp through many more tiles than the uncapped grid does."""
import numpy as np
import pytest
import torch

import quantized_tensor_activation_gb300 as qta
from gpu_util import device, random_values, to_dtype_cpu

pytestmark = pytest.mark.gpu


def _step(scheme, B, gscheme, gB, x, n, rows, cols, max_sms):
    dev = x.device
    d_in = qta.desc(scheme, B, rows, cols, batch=n, max_sms=max_sms)
    q = qta.alloc_qtensor(d_in, dev)
    qta.taco_compress(d_in, x, qta.BF16, q, qta.SCALE_CURRENT)
    d_sh = qta.desc(scheme, B, rows, cols, max_sms=max_sms)
    d_g = qta.desc(gscheme, gB, rows // n, cols, batch=n, max_sms=max_sms)
    g = qta.alloc_qtensor(d_g, dev)
    shards = [q.shard(r) for r in range(n)]
    qta.qar_reduce_requant(d_sh, shards, 0, rows, d_g, g, qta.SCALE_CURRENT)
    s = torch.empty((rows, cols), dtype=torch.float32, device=dev)
    qta.qar_reduce(d_sh, shards, 0, rows, s)
    y = torch.empty((rows, cols), dtype=torch.bfloat16, device=dev)
    qta.taco_decompress(d_g, g, y, qta.BF16)
    h = torch.empty((rows, cols), dtype=torch.float32, device=dev)
    qta.qar_dequant_add(d_g, g, y, qta.BF16, h)
    # the shards themselves decompressed: with one or seven SMs every warp's
    # stage ring wraps many times (INT4 included)
    xq = torch.empty((n, rows, cols), dtype=torch.bfloat16, device=dev)
    qta.taco_decompress(d_in, q, xq, qta.BF16)
    torch.cuda.synchronize()
    out = [q.codes, q.scales, g.codes, g.scales, s, y, h, xq]
    return [t.clone() for t in out if t is not None]


@pytest.mark.parametrize("scheme,B,gscheme,gB", [("taco_fp8", 128, "taco_fp8", 128),
                                                  ("int4_asym", 128, "int8_asym", 128)])
@pytest.mark.parametrize("n,rows", [(4, 96), (5, 120)])   # 5: a stage of the INT4 reduce holds a lone rank
def test_same_bytes_with_fewer_sms(scheme, B, gscheme, gB, n, rows):
    dev = device()
    cols = 1024
    x = to_dtype_cpu(random_values(np.random.default_rng(2), (n, rows, cols), "mixed"), qta.BF16).to(dev)
    ref = _step(scheme, B, gscheme, gB, x, n, rows, cols, 0)
    for m in (1, 7):
        got = _step(scheme, B, gscheme, gB, x, n, rows, cols, m)
        for a, b in zip(ref, got):
            assert torch.equal(a.view(torch.uint8) if a.dtype != torch.uint8 else a,
                               b.view(torch.uint8) if b.dtype != torch.uint8 else b)
    assert qta.qta_device_error() == 0
