"""Checks of the oracle against the values the pages print (fixtures under
tests/golden/, each with its citation)."""
import os

import numpy as np

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read(name):
    vals = {}
    for line in open(os.path.join(HERE, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            vals[k] = float(v)
    return vals


def test_eq3_ulp_bound_from_the_printed_formula(orc):
    g = _read("taco_eq3_fp8_ulp.txt")
    m, top = int(g["mantissa_bits"]), g["max_finite"]
    assert orc.e4m3_decode(np.array([0x7E], np.uint8))[0] == top     # the format's largest finite value
    rng = np.random.default_rng(8)
    v = np.exp2(rng.uniform(-6, np.log2(top), 500_000)).astype(np.float32)
    q = orc.e4m3_decode(orc.e4m3_encode(v)).astype(np.float64)
    ulp = np.exp2(np.floor(np.log2(v.astype(np.float64))) - m)
    assert np.all(np.abs(v - q) <= ulp)


def test_ring_allreduce_mse_near_equarx_figures(orc):
    """Our reading of the adder chains (8 ranks, INT8 B64, N(0,1)) against the
    printed MSEs.  The pages do not give the ring size or topology, so this is
    a consistency check within 25 %, not a bit pin."""
    g = _read("equarx_allreduce_mse.txt")
    rng = np.random.default_rng(0)
    n, rows, cols = 8, 64, 1024
    xs = [orc.f32_to_bf16(rng.standard_normal(rows * cols).astype(np.float32)) for _ in range(n)]
    xw = [orc.bf16_to_f32(x).astype(np.float64) for x in xs]
    exact = sum(xw)
    got = {}
    for name, semi in (("full_loop", False), ("semi_loop", True)):
        _, y = orc.ring_allreduce(orc.INT8_SYM, 64, xs, orc.BF16, rows, cols, semi)
        got[name] = float(((y - exact) ** 2).mean())
    acc = np.zeros(rows * cols, np.float32)
    for x in xw:
        acc = (acc + x.astype(np.float32)).astype(np.float32)       # unquantized reduce-scatter
    c, s, z = orc.compress(orc.INT8_SYM, 64, acc, orc.FP32, 1, rows, cols, None, orc.CURRENT)
    y = orc.decompress(orc.INT8_SYM, 64, c, s, z, None, 1, rows, cols, orc.FP32)
    got["allgather_only"] = float(((y - exact) ** 2).mean())
    for k, ref in g.items():
        assert 0.75 <= got[k] / ref <= 1.25, (k, got[k], ref)
    assert got["full_loop"] > got["semi_loop"] > got["allgather_only"]
