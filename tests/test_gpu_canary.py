"""Guard bytes around every output: each call writes exactly its outputs.
Every output buffer (codes, scales, zeros, per-tensor state, FP32 sums,
decompressed values) sits inside a larger allocation filled with a canary
pattern; after the calls on ragged shapes (partial last warp tile, tensor
boundaries inside a tile) the guard regions must be unchanged.  This stands
in for a memory checker: the TMA stores clip at their tensor maps and the
plain stores are guarded by index, and this test checks both."""
import numpy as np
import pytest
import torch

import quantized_tensor_activation_gb300 as qta
from gpu_util import device, random_values, to_dtype_cpu

pytestmark = pytest.mark.gpu

PAD = 4096          # guard bytes on each side (a multiple of 256: keeps every view aligned)
CANARY = 0xA5


class Guarded:
    """Byte buffers with PAD canary bytes on both sides; views are the payloads."""

    def __init__(self, dev):
        self.dev = dev
        self.bufs = []

    def bytes(self, n):
        raw = torch.full((n + 2 * PAD,), CANARY, dtype=torch.uint8, device=self.dev)
        self.bufs.append((raw, n))
        return raw[PAD:PAD + n]

    def floats(self, n, fill=None):
        v = self.bytes(4 * n).view(torch.float32)
        if fill is not None:
            v.copy_(torch.as_tensor(fill, dtype=torch.float32))
        return v

    def qtensor(self, d, scale=1.0):
        cb, sb, zb, stb = qta.codes_bytes(d), qta.scales_bytes(d), qta.zeros_bytes(d), qta.state_bytes(d)
        st = None
        if stb:
            init = np.zeros(stb // 4, dtype=np.float32)
            init[0::2] = scale
            st = self.floats(stb // 4, init)
        return qta.QTensor(d, self.bytes(cb), self.bytes(sb), self.bytes(zb) if zb else None, st)

    def check(self):
        torch.cuda.synchronize()
        for raw, n in self.bufs:
            head, tail = raw[:PAD], raw[PAD + n:]
            assert bool((head == CANARY).all()) and bool((tail == CANARY).all()), f"guard overwritten ({n} B)"


CASES = [("taco_fp8", 128, "taco_fp8", 128), ("taco_fp8", 256, "taco_fp8", 64), ("taco_fp8", 64, "taco_fp8", 256),
         ("int8_sym", 64, "int8_sym", 64), ("int4_asym", 128, "int8_asym", 128),
         ("int8_asym", 128, "int8_asym", 128)]


@pytest.mark.parametrize("scheme,B,gscheme,gB", CASES)
def test_every_call_writes_only_its_outputs(scheme, B, gscheme, gB):
    dev = device()
    g = Guarded(dev)
    n, rows, cols = 3, 14, 768                       # 3*14*768/64 = 504 segments: 15.75 warp tiles
    rng = np.random.default_rng(B + len(scheme))
    x = to_dtype_cpu(random_values(rng, (n, rows, cols), "mixed"), qta.BF16).to(dev)
    d_in = qta.desc(scheme, B, rows, cols, batch=n)
    q = g.qtensor(d_in)
    qta.taco_compress(d_in, x, qta.BF16, q, qta.SCALE_CURRENT)
    d_sh = qta.desc(scheme, B, rows, cols)
    shards = [q.shard(r) for r in range(n)]
    s = g.floats(rows * cols)
    qta.qar_reduce(d_sh, shards, 0, rows, s)
    s_part = g.floats(5 * cols)
    qta.qar_reduce(d_sh, shards, 3, 8, s_part)                     # a row range
    d_g = qta.desc(gscheme, gB, 7, cols, batch=2)                  # 14 rows as 2 shards of 7
    gq = g.qtensor(d_g, 0.01)
    qta.qar_reduce_requant(d_sh, shards, 0, rows, d_g, gq, qta.SCALE_CURRENT)
    gq2 = g.qtensor(d_g, 0.01)
    qta.qar_requant(d_g, s, gq2, qta.SCALE_DELAYED)
    y = g.bytes(2 * rows * cols).view(torch.bfloat16)
    qta.taco_decompress(d_g, gq, y, qta.BF16)
    yf = g.floats(rows * cols)
    qta.taco_decompress(d_g, gq2, yf, qta.FP32)
    h = g.floats(rows * cols)
    qta.qar_dequant_add(d_g, gq, y, qta.BF16, h)
    gq3 = g.qtensor(d_g, 0.01)
    qta.qar_dequant_add_requant(d_g, gq, yf, qta.FP32, gq3, qta.SCALE_CURRENT)
    e = g.bytes(8).view(torch.float64)
    qta.qta_sq_error(y, qta.BF16, yf, rows * cols, e)
    if q.state is not None:
        qta.taco_update_scale(q.state, n)
    g.check()
    assert qta.qta_device_error() == 0


def test_rescaling_calls_write_only_their_outputs():
    # the channel amax writes only the amax part of the state; the update
    # writes the state; the codec calls with the factors write their outputs
    dev = device()
    g = Guarded(dev)
    n, rows, cols = 3, 14, 768
    rng = np.random.default_rng(5)
    x = to_dtype_cpu(random_values(rng, (n, rows, cols), "mixed"), qta.BF16).to(dev)
    raw = torch.full((3 * cols * 4 + 2 * PAD,), CANARY, dtype=torch.uint8, device=dev)
    chan = raw[PAD:PAD + 3 * cols * 4].view(torch.float32)
    chan[:2 * cols] = 1.0
    chan[2 * cols:] = 0.0
    fill = raw[PAD:PAD + 2 * cols * 4].clone()
    d_in = qta.desc("taco_fp8", 128, rows, cols, batch=n)
    qta.taco_channel_amax(d_in, x, qta.BF16, chan)
    torch.cuda.synchronize()
    assert torch.equal(raw[PAD:PAD + 2 * cols * 4], fill)           # down and up untouched
    qta.taco_ash_update(chan, cols)
    torch.cuda.synchronize()
    assert bool((raw[:PAD] == CANARY).all()) and bool((raw[PAD + 3 * cols * 4:] == CANARY).all())
    q = g.qtensor(d_in)
    q.chan = chan
    qta.taco_compress(d_in, x, qta.BF16, q, qta.SCALE_CURRENT)
    d_sh = qta.desc("taco_fp8", 128, rows, cols)
    shards = [q.shard(r) for r in range(n)]
    s = g.floats(rows * cols)
    qta.qar_reduce(d_sh, shards, 0, rows, s)
    d_g = qta.desc("taco_fp8", 256, 7, cols, batch=2)
    gq = g.qtensor(d_g, 0.01)
    gq.chan = chan
    qta.qar_reduce_requant(d_sh, shards, 0, rows, d_g, gq, qta.SCALE_CURRENT)
    y = g.bytes(2 * rows * cols).view(torch.bfloat16)
    qta.taco_decompress(d_g, gq, y, qta.BF16)
    g.check()
    assert bool((raw[:PAD] == CANARY).all()) and bool((raw[PAD + 3 * cols * 4:] == CANARY).all())
    assert qta.qta_device_error() == 0
