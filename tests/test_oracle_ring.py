"""Oracle pins for the ring hop (dequantize the incoming partial sum, add the
local tensor) and the adder chains built from it ([EQuARX] What carries the
argument; Figs. 4-5, full-loop and semi-loop adder chains)."""
import numpy as np
import pytest

SCHEMES = [("taco", 0, 128), ("int8", 1, 64), ("int4", 2, 128), ("int8a", 3, 128)]


def _quantized(orc, scheme, B, rng, rows, cols):
    x = rng.standard_normal(rows * cols).astype(np.float32)
    st = np.zeros(2, np.float32) if scheme == orc.TACO_FP8 else None
    c, s, z = orc.compress(scheme, B, x, orc.FP32, 1, rows, cols, st, orc.CURRENT)
    return c, s, z, st


@pytest.mark.parametrize("name,scheme,B", SCHEMES)
@pytest.mark.parametrize("xdt", ["bf16", "fp16", "fp32"])
def test_dequant_add_is_one_fp32_addition(orc, name, scheme, B, xdt):
    rng = np.random.default_rng(11)
    rows, cols = 4, 512
    q = _quantized(orc, scheme, B, rng, rows, cols)
    xv = rng.standard_normal(rows * cols).astype(np.float32)
    if xdt == "bf16":
        xb, dt = orc.f32_to_bf16(xv), orc.BF16
        xw = orc.bf16_to_f32(xb)
    elif xdt == "fp16":
        xb, dt = orc.f32_to_f16(xv), orc.FP16
        xw = orc.f16_to_f32(xb)
    else:
        xb, dt, xw = xv, orc.FP32, xv
    got = orc.dequant_add(scheme, B, *q, 1, rows, cols, xb, dt)
    deq = orc.decompress(scheme, B, *q, 1, rows, cols, orc.FP32)
    # two FP32 values of similar magnitude add exactly in float64; one
    # rounding of that exact sum to float32 is the IEEE addition
    want = (deq.astype(np.float64) + xw.astype(np.float64)).astype(np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_chain_orders():
    import oracle as orc
    assert orc.ring_chunk_orders(8, 0, False) == [[1, 2, 3, 4, 5, 6, 7]]
    assert orc.ring_chunk_orders(8, 0, True) == [[4, 3, 2, 1], [5, 6, 7]]
    assert orc.ring_chunk_orders(8, 5, True) == [[1, 0, 7, 6], [2, 3, 4]]
    assert orc.ring_chunk_orders(2, 1, True) == [[0]]
    for n in (2, 3, 4, 7, 8):
        for j in range(n):
            for semi in (False, True):
                chains = orc.ring_chunk_orders(n, j, semi)
                seen = sorted(r for c in chains for r in c)
                assert seen == sorted(set(range(n)) - {j})   # every other rank once
                for c in chains:                                 # each chain walks to the owner
                    assert (c[-1] - j) % n in (1, n - 1)


def _exact_int8_inputs(n, rows, cols, semi, rng):
    """Integer inputs for which every partial sum on every chain has block
    absmax exactly 127, so every INT8 scale is 1 and every hop is exact."""
    rc = rows // n
    xs = rng.integers(-3, 4, size=(n, rows, cols)).astype(np.float32)
    xs[:, :, 0::64] = 0.0
    xs[:, :, 1::64] = 0.0
    import oracle as orc
    for j in range(n):
        for k, chain in enumerate(orc.ring_chunk_orders(n, j, semi)):
            xs[chain[0], j * rc:(j + 1) * rc, k::64] = 127.0   # the chain's first rank
    return xs


@pytest.mark.parametrize("semi", [False, True])
@pytest.mark.parametrize("n", [2, 3, 8])
def test_int8_chain_exact_when_every_partial_is_representable(orc, semi, n):
    rng = np.random.default_rng(5)
    rows, cols = 2 * n, 256
    xs = _exact_int8_inputs(n, rows, cols, semi, rng)
    bits = [orc.f32_to_bf16(x.reshape(-1)) for x in xs]
    s = orc.ring_reduce_scatter(orc.INT8_SYM, 64, bits, orc.BF16, rows, cols, semi)
    assert np.array_equal(s, xs.sum(axis=0).reshape(-1))


@pytest.mark.parametrize("name,scheme,B", SCHEMES)
def test_two_ranks_full_equals_semi(orc, name, scheme, B):
    rng = np.random.default_rng(7)
    xs = [orc.f32_to_bf16(rng.standard_normal(8 * 256).astype(np.float32)) for _ in range(2)]
    a = orc.ring_allreduce(scheme, B, xs, orc.BF16, 8, 256, semi=False)
    b = orc.ring_allreduce(scheme, B, xs, orc.BF16, 8, 256, semi=True)
    assert np.array_equal(a[0].view(np.uint32), b[0].view(np.uint32))
    assert np.array_equal(a[1].view(np.uint32), b[1].view(np.uint32))


def test_error_grows_with_hops_and_semi_loop_is_shorter(orc):
    rng = np.random.default_rng(3)
    n, rows, cols = 8, 64, 1024
    xf = [rng.standard_normal(rows * cols).astype(np.float32) for _ in range(n)]
    xs = [orc.f32_to_bf16(x) for x in xf]
    xw = [orc.bf16_to_f32(x).astype(np.float64) for x in xs]
    exact = sum(xw)
    # partial sums of one chain after k ranks: error grows with the hops
    mse = []
    for k in range(1, n):
        q = orc.ring_chain(orc.INT8_SYM, 64, xs[:k], orc.BF16, rows, cols)
        p = orc.decompress(orc.INT8_SYM, 64, *q, 1, rows, cols, orc.FP32).astype(np.float64)
        mse.append(float(((p - sum(xw[:k])) ** 2).mean()))
    assert all(b > a for a, b in zip(mse, mse[1:])), mse
    full = orc.ring_reduce_scatter(orc.INT8_SYM, 64, xs, orc.BF16, rows, cols, semi=False)
    semi = orc.ring_reduce_scatter(orc.INT8_SYM, 64, xs, orc.BF16, rows, cols, semi=True)
    e_full = float(((full - exact) ** 2).mean())
    e_semi = float(((semi - exact) ** 2).mean())
    assert e_semi < 0.8 * e_full, (e_full, e_semi)
