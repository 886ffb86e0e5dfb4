"""Pins of the oracle's codecs and reduction against definitions, brute force,
closed forms and bounds (not against retyped formulas).

TACO (dual-scale FP8 after the block Hadamard; TACO Core claim, Fig. 7):
  * exact round trip of blocks whose transform is E4M3-representable with
    absmax 448 (then S = r_b = s_b = 1);
  * every code is the nearest of the 256 E4M3 codes to y / s_b (searched),
    every scale byte the nearest code to a_b / (448 S) (searched);
  * the per-tensor scale follows amax / 448 of the exact (int64) transform;
  * reconstruction error obeys Eq. (3) (TACO Fig. 6) mapped through the
    orthogonal inverse transform.
EQuARX int8 (one FP32 scale per 64, dequantize to FP32 before adding):
  * integer blocks with absmax 127 round-trip exactly; codes are the nearest
    integers; |x - q s| <= s/2.
Flash Communication asymmetric group-128 INT4/INT8:
  * scale and zero are numpy's float16 roundings of (max-min)/Q and min;
  * codes are the nearest grid points (searched); nibble order is checked on
    a group whose codes are known in advance; exact round trip on grid data.
Reduce: equals the float64 sum of per-rank dequantized values within the
FP32 bound, N = 1 equals the decompression, rank order changes the sum only
within that bound.
"""
import numpy as np
import pytest
import scipy.linalg

import workloads


def _bf16(orc, x):
    return orc.f32_to_bf16(np.asarray(x, dtype=np.float32))


def _e4m3_pos():
    import torch
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float32).numpy()


def _nearest_codes(v, table):
    """Brute force over all codes: indices of all codes at minimal distance."""
    fin = ~np.isnan(table)
    d = np.abs(v[:, None].astype(np.float64) - np.where(fin, table, np.inf)[None, :].astype(np.float64))
    m = d.min(axis=1, keepdims=True)
    return d <= m * (1 + 1e-12) + 1e-300


# --------------------------------------------------------------------- TACO
def test_taco_exact_roundtrip(orc):
    B = 128
    rng = np.random.default_rng(0)
    rows = []
    for _ in range(16):
        x = np.zeros(B, dtype=np.float32)
        j, k = rng.choice(B, 2, replace=False)
        x[j] = 224.0
        x[k] = 224.0 * rng.choice([-1, 1])   # transform entries in {0, +-448}
        rows.append(x)
    x = np.concatenate(rows)
    xb = _bf16(orc, x)
    st = np.zeros(2, dtype=np.float32)
    codes, scales, _ = orc.compress(orc.TACO_FP8, B, xb, orc.BF16, 1, 16, B, st, orc.CURRENT)
    assert st[0] == 1.0 and st[1] == 448.0
    assert np.all(scales == 0x38)                       # r_b = 1.0
    y = orc.decompress(orc.TACO_FP8, B, codes, scales, None, st, 1, 16, B, orc.BF16)
    assert np.array_equal(y, xb)


@pytest.mark.parametrize("B", [4, 8, 64, 128, 256])
def test_taco_codes_and_scales_are_nearest(orc, B):
    rng = np.random.default_rng(B)
    nb = 64 if B <= 8 else 24
    xi = rng.integers(-60, 61, size=(nb, B))
    xi[::5] *= 9                                         # some large blocks
    xi[3] = 0                                            # an all-zero block
    x = xi.astype(np.float32).reshape(-1)
    # delayed scale from a (deliberately stale) previous step
    S = np.float32(7.3)
    st = np.array([S, 0.0], dtype=np.float32)
    codes, scales, _ = orc.compress(orc.TACO_FP8, B, x, orc.FP32, 1, nb, B, st, orc.DELAYED)
    y = (xi @ scipy.linalg.hadamard(B).T).astype(np.float64)          # exact
    a = np.abs(y).max(axis=1)
    assert st[1] == np.float32(a.max())
    table = _e4m3_pos()
    r = table[scales].astype(np.float64)
    # scale byte: nearest code to a_b / (448 S), with r_b forced to 2^-9 when it would be 0
    ratio = a / (448.0 * float(S))
    ok = _nearest_codes(ratio, table)[np.arange(nb), scales]
    ok |= (scales == 1) & (a > 0) & (ratio < 2.0 ** -10)
    ok |= (a == 0) & (scales == 0)
    assert np.all(ok)
    sb = (np.float32(S) * table[scales]).astype(np.float64)
    c = codes.reshape(nb, B)
    for b in range(nb):
        if sb[b] == 0:
            assert np.all((c[b] & 0x7F) == 0)
            continue
        v = y[b] / sb[b]
        near = _nearest_codes(np.clip(v, -448, 448), table)
        assert np.all(near[np.arange(B), c[b]]), b
        # saturation rule: exactly the values past 464 land on +-448 by clipping
        sat = np.abs(v) >= 464
        assert np.all((c[b][sat] & 0x7F) == 0x7E)


@pytest.mark.parametrize("B", [4, 64, 128, 256])
@pytest.mark.parametrize("mode_name", ["DELAYED", "CURRENT"])
def test_taco_round_up_scales_are_the_smallest_cover(orc, B, mode_name):
    """QTA_SCALE_ROUND_UP: the scale byte is the smallest E4M3 code whose
    value is not below a_b / (448 S) (searched over the table, ratio in
    float64 from the exact integer transform), and with a current S no code
    saturates."""
    rng = np.random.default_rng(40 + B)
    nb = 48
    xi = rng.integers(-60, 61, size=(nb, B))
    xi[::5] *= 9
    xi[3] = 0
    x = xi.astype(np.float32).reshape(-1)
    mode = getattr(orc, mode_name) | orc.ROUND_UP
    st = np.array([7.3, 0.0], dtype=np.float32)
    codes, scales, _ = orc.compress(orc.TACO_FP8, B, x, orc.FP32, 1, nb, B, st, mode)
    y = (xi @ scipy.linalg.hadamard(B).T).astype(np.float64)
    a = np.abs(y).max(axis=1)
    S = float(st[0])
    table = _e4m3_pos()
    ratio = a / (448.0 * S)
    pos = table[:0x7F].astype(np.float64)                 # +0 .. 448
    for b in range(nb):
        if a[b] == 0:
            assert scales[b] == 0
            continue
        cover = np.nonzero(pos >= ratio[b] * (1 - 2.0 ** -22))[0]
        want = cover[0] if cover.size else 0x7E
        # the FP32 ratio may sit a rounding away from the float64 one
        assert scales[b] in (want, want + 1) and table[scales[b]] >= ratio[b] * (1 - 2.0 ** -22), b
        if scales[b] == want + 1:
            assert abs(pos[want] / ratio[b] - 1) < 2.0 ** -20
    if mode_name == "CURRENT":
        sb = (np.float32(S) * table[scales]).astype(np.float64)
        v = np.abs(y) / np.where(sb > 0, sb, 1.0)[:, None]
        assert v.max() <= 448.0 * (1 + 2.0 ** -20)
        assert not np.any((codes.reshape(nb, B) & 0x7F) == 0x7F)


def test_taco_round_up_never_below_nearest(orc):
    rng = np.random.default_rng(9)
    x = (rng.standard_normal(64 * 128) * np.exp(rng.uniform(-3, 3, 64 * 128))).astype(np.float32)
    s1 = np.zeros(2, np.float32)
    s2 = np.zeros(2, np.float32)
    _, near, _ = orc.compress(orc.TACO_FP8, 128, x, orc.FP32, 1, 64, 128, s1, orc.CURRENT)
    _, up, _ = orc.compress(orc.TACO_FP8, 128, x, orc.FP32, 1, 64, 128, s2, orc.CURRENT | orc.ROUND_UP)
    assert s1[0] == s2[0]
    assert np.all((up == near) | (up == near + 1))
    assert np.any(up == near + 1) and np.any(up == near)


def test_taco_current_scale_rule(orc):
    w = workloads.WORKLOADS["taco_tiny"]
    import torch
    xt = workloads.make_rank_inputs(w, rows=32, ranks=2)
    xb = xt.view(torch.int16).numpy().view(np.uint16).reshape(-1)
    st = np.zeros(4, dtype=np.float32)
    orc.compress(orc.TACO_FP8, 128, xb, orc.BF16, 2, 32, 1024, st, orc.CURRENT)
    xf = xt.float().numpy().reshape(2, -1, 128).astype(np.float64)
    y = xf @ scipy.linalg.hadamard(128).T
    for t in range(2):
        amax = np.abs(y[t]).max()
        assert abs(st[2 * t + 1] - amax) <= 1e-6 * amax
        assert st[2 * t] == np.float32(np.float32(st[2 * t + 1]) / np.float32(448.0))
    # update: S <- amax/448, amax <- 0; degenerate amax falls back to 1
    s2 = st.copy()
    orc.taco_update_scale(s2)
    assert s2[1] == 0 and s2[3] == 0 and s2[0] == st[0]
    z = np.array([1.0, 0.0, 1.0, np.inf, 1.0, np.nan, 1.0, 1e-45], dtype=np.float32)
    orc.taco_update_scale(z)
    assert list(z[0::2]) == [1.0, 1.0, 1.0, 1.0]


@pytest.mark.parametrize("B", [128, 256])
def test_taco_reconstruction_within_eq3(orc, B):
    # Error in the Hadamard domain is at most half an E4M3 ULP of y/s_b times
    # s_b (Eq. 3), or the clipping at 448 for saturated values; the inverse
    # transform H/B is orthogonal up to 1/sqrt(B), so ||x - x^||_2 <=
    # ||e||_2 / sqrt(B), plus the final bf16 rounding.
    w = workloads.WORKLOADS["taco_tiny"]
    import torch
    xt = workloads.make_rank_inputs(w, rows=16, ranks=1)
    xb = xt.view(torch.int16).numpy().view(np.uint16).reshape(-1)
    st = np.zeros(2, dtype=np.float32)
    codes, scales, _ = orc.compress(orc.TACO_FP8, B, xb, orc.BF16, 1, 16, 1024, st, orc.CURRENT)
    yf = orc.decompress(orc.TACO_FP8, B, codes, scales, None, st, 1, 16, 1024, orc.FP32)
    x = xt.float().numpy().reshape(-1, B).astype(np.float64)
    y = x @ scipy.linalg.hadamard(B).T
    table = _e4m3_pos()
    sb = (np.float32(st[0]) * table[scales]).astype(np.float64)[:, None]
    v = np.abs(y) / sb
    ulp = np.exp2(np.floor(np.log2(np.maximum(v, 2.0 ** -6))) - 3)
    e_h = np.where(v > 448, v - 448, ulp / 2) * sb
    bound = np.sqrt((e_h ** 2).sum(axis=1)) / np.sqrt(B) * 1.001 + 1e-6 * np.abs(x).max(axis=1)
    err = np.sqrt(((yf.reshape(-1, B) - x) ** 2).sum(axis=1))
    assert np.all(err <= bound)


# --------------------------------------------------------------------- INT8
def test_int8_sym_exact_and_nearest(orc):
    rng = np.random.default_rng(5)
    xi = rng.integers(-127, 128, size=(40, 64))
    xi[:, 7] = 127
    codes, scales, _ = orc.compress(orc.INT8_SYM, 64, xi.astype(np.float32).reshape(-1), orc.FP32, 1, 40, 64)
    assert np.all(scales == 1.0) and np.array_equal(codes.reshape(40, 64), xi.astype(np.int8))
    x = (rng.standard_normal((300, 64)) * np.exp(rng.uniform(-5, 5, (300, 1)))).astype(np.float32)
    x[4] = 0
    codes, scales, _ = orc.compress(orc.INT8_SYM, 64, x.reshape(-1), orc.FP32, 1, 300, 64)
    a = np.abs(x).max(axis=1).astype(np.float64)
    assert np.allclose(scales, a / 127, rtol=1e-7, atol=0)
    q = codes.reshape(300, 64).astype(np.float64)
    t = np.where(a[:, None] > 0, x * 127.0 / np.where(a[:, None] > 0, a[:, None], 1), 0)
    assert np.all(np.abs(q - t) <= 0.5 + 1e-5)
    assert np.all(np.abs(q) <= 127)
    deq = orc.decompress(orc.INT8_SYM, 64, codes, scales, None, None, 1, 300, 64, orc.FP32).reshape(300, 64)
    assert np.all(np.abs(deq - x) <= scales[:, None].astype(np.float64) * (0.5 + 1e-5))
    assert np.all(deq[4] == 0)


# --------------------------------------------------------------------- ASYM
@pytest.mark.parametrize("bits", [4, 8])
def test_asym_scale_zero_codes(orc, bits):
    scheme = orc.INT4_ASYM if bits == 4 else orc.INT8_ASYM
    Q = 2 ** bits - 1
    rng = np.random.default_rng(bits)
    x = (rng.standard_t(3, size=(80, 128)) * np.exp(rng.uniform(-4, 3, (80, 1)))).astype(np.float16)
    x[5] = 1.5                                          # constant group: s = 0
    xb = x.view(np.uint16).reshape(-1)
    codes, scales, zeros = orc.compress(scheme, 128, xb, orc.FP16, 1, 80, 128)
    xf = x.astype(np.float32)
    mn, mx = xf.min(axis=1), xf.max(axis=1)
    s_ref = np.minimum((mx - mn) / np.float32(Q), np.float32(65504)).astype(np.float16)
    assert np.array_equal(scales, s_ref.view(np.uint16))
    assert np.array_equal(zeros, mn.astype(np.float16).view(np.uint16))
    if bits == 4:
        q = np.stack([codes & 15, codes >> 4], axis=1).reshape(80, 128)
    else:
        q = codes.reshape(80, 128)
    s = s_ref.astype(np.float32)
    z = mn.astype(np.float16).astype(np.float32)
    grid = np.arange(Q + 1, dtype=np.float64)
    for g in range(80):
        if s[g] == 0:
            assert np.all(q[g] == 0)
            continue
        d = np.abs(xf[g][:, None].astype(np.float64) - (z[g] + grid[None, :] * s[g]))
        best = d.min(axis=1, keepdims=True)
        hit = d[np.arange(128), q[g]]
        assert np.all(hit <= best[:, 0] + 1e-6 * s[g])
    deq = orc.decompress(scheme, 128, codes, scales, zeros, None, 1, 80, 128, orc.FP32).reshape(80, 128)
    assert np.all(np.abs(deq - xf) <= s[:, None] * (0.5 + 1e-4) + 1e-7)


def test_int4_nibble_order_and_exact_grid(orc):
    q = np.tile(np.arange(16), 8)                        # 128 known codes
    x = (q * 0.25 - 1.0).astype(np.float32)              # min -1, step 0.25
    codes, scales, zeros = orc.compress(orc.INT4_ASYM, 128, x, orc.FP32, 1, 1, 128)
    expect = (q[0::2] | (q[1::2] << 4)).astype(np.uint8)
    assert np.array_equal(codes, expect)
    assert scales[0] == np.float16(0.25).view(np.uint16) and zeros[0] == np.float16(-1.0).view(np.uint16)
    y = orc.decompress(orc.INT4_ASYM, 128, codes, scales, zeros, None, 1, 1, 128, orc.FP32)
    assert np.array_equal(y, x)


# --------------------------------------------------------------------- reduce
def _make_shards(orc, scheme, B, n, rows, cols, seed=0):
    rng = np.random.default_rng(seed)
    shards, deq = [], []
    for r in range(n):
        x = (rng.standard_normal((rows, cols)) * (1 + r)).astype(np.float32).reshape(-1)
        st = np.zeros(2, dtype=np.float32) if scheme == orc.TACO_FP8 else None
        c, s, z = orc.compress(scheme, B, x, orc.FP32, 1, rows, cols, st, orc.CURRENT)
        shards.append((c, s, z, st))
        deq.append(orc.decompress(scheme, B, c, s, z, st, 1, rows, cols, orc.FP32))
    return shards, deq


@pytest.mark.parametrize("scheme,B", [(0, 128), (0, 256), (1, 64), (2, 128), (3, 128)])
def test_reduce_matches_float64_sum(orc, scheme, B):
    n, rows, cols = 5, 12, 512
    shards, deq = _make_shards(orc, scheme, B, n, rows, cols)
    out = orc.reduce(scheme, B, shards, rows, cols)
    if scheme == orc.TACO_FP8:
        # dequantized values in the Hadamard domain, summed in float64, then the
        # exact float64 inverse transform
        table = _e4m3_pos().astype(np.float64)
        H = scipy.linalg.hadamard(B).astype(np.float64)
        acc = np.zeros((rows * cols // B, B))
        mag = np.zeros_like(acc)
        for c, s, z, st in shards:
            sb = (np.float32(st[0]) * table[s].astype(np.float32)).astype(np.float64)
            v = table[c].reshape(-1, B) * sb[:, None]
            acc += v
            mag += np.abs(v)
        ref = (acc @ H.T / B).reshape(-1)
        bound = ((n + np.log2(B)) * 2.0 ** -24 * (mag @ np.abs(H).T / B)).reshape(-1) * 1.01
    else:
        d = np.stack(deq).astype(np.float64)
        ref = d.sum(axis=0)
        bound = n * 2.0 ** -24 * np.abs(d).sum(axis=0) * 1.01
    assert np.all(np.abs(out - ref) <= bound + 1e-30)
    # N = 1 reduces to the decompression (FP32 output)
    one = orc.reduce(scheme, B, shards[:1], rows, cols)
    assert np.array_equal(one, deq[0])
    # rank order changes the sum only within the bound
    perm = orc.reduce(scheme, B, shards[::-1], rows, cols)
    assert np.all(np.abs(perm - ref) <= bound + 1e-30)
    # a row range gives the same rows as the full reduction
    part = orc.reduce(scheme, B, shards, rows, cols, 3, 7)
    assert np.array_equal(part, out[3 * cols:7 * cols])


def _round_f32(x):
    """Exact rational -> nearest binary32 (ties to even), by integer arithmetic."""
    from fractions import Fraction
    if x == 0:
        return 0.0
    sign = -1 if x < 0 else 1
    a = abs(Fraction(x))
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126) - 23                     # grid step 2^e (subnormals: 2^-149)
    q = a / Fraction(2) ** e
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * float(n * Fraction(2) ** e)


@pytest.mark.parametrize("scheme,B", [(0, 128), (1, 64)])
def test_reduce_accumulates_with_one_rounding_per_rank(orc, scheme, B):
    # rank-order sum: acc = RN(c0*s0), then acc = RN(c1*s1 + acc) with the product exact
    # (a fused multiply-add); emulated here with exact rationals.
    from fractions import Fraction
    rows, cols = 2, 256
    shards, _ = _make_shards(orc, scheme, B, 3, rows, cols, seed=9)
    out = orc.reduce(scheme, B, shards, rows, cols)
    table = _e4m3_pos()
    E = rows * cols
    acc = np.zeros(E, dtype=np.float64)
    for e in range(E):
        a = None
        for r, (c, s, z, st) in enumerate(shards):
            if scheme == orc.TACO_FP8:
                code = Fraction(float(table[c[e]]))
                sc = Fraction(float(np.float32(st[0]) * table[s[e // B]]))
            else:
                code = Fraction(int(c[e]))
                sc = Fraction(float(s[e // 64]))
            a = _round_f32(code * sc) if r == 0 else _round_f32(code * sc + Fraction(a))
        acc[e] = a
    ref = acc.astype(np.float32)
    if scheme == orc.TACO_FP8:
        ref = (orc.fwht(ref, B) * np.float32(1.0 / B)).astype(np.float32)
    assert np.array_equal(out.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("scheme,B,oscheme,oB", [(1, 64, 1, 64), (2, 128, 3, 128), (3, 128, 3, 128),
                                                 (0, 128, 0, 256), (0, 256, 0, 64)])
def test_reduce_requant_equals_two_calls(orc, scheme, B, oscheme, oB):
    # every pair but TACO -> TACO with equal blocks is reduce, then compress
    rows, cols, n = 16, 512, 3
    shards, _ = _make_shards(orc, scheme, B, n, rows, cols, seed=21)
    st1 = np.array([0.01, 0.0, 0.02, 0.1], dtype=np.float32)
    st2 = st1.copy()
    f = orc.reduce_requant(scheme, B, shards, rows, cols, 2, 10, oscheme, oB, 2, st1 if oscheme == 0 else None)
    s = orc.reduce(scheme, B, shards, rows, cols, 2, 10)
    c = orc.compress(oscheme, oB, s, orc.FP32, 2, 4, cols, st2 if oscheme == 0 else None)
    for a, b in zip(f, c):
        assert (a is None and b is None) or np.array_equal(a, b)
    assert np.array_equal(st1, st2)


@pytest.mark.parametrize("mode", [0, 1])
def test_reduce_requant_taco_hadamard_domain(orc, mode):
    # TACO -> TACO, equal blocks: the codes quantize the exact FP32 Hadamard-
    # domain sums (emulated with exact rationals) -- every code is the nearest
    # E4M3 value to sum/s_b and every block byte the nearest to a_b/(448 S) --
    # and decompressing them approximates the float64 sum of the inputs within
    # the FP8 error of Eq. (3) (TACO Fig. 6).
    from fractions import Fraction
    B, rows, cols, n = 128, 2, 256, 3
    shards, deq = _make_shards(orc, 0, B, n, rows, cols, seed=5)
    st = np.array([0.02, 0.0], dtype=np.float32)
    c, s, _ = orc.reduce_requant(0, B, shards, rows, cols, 0, rows, 0, B, 1, st, mode)
    table = _e4m3_pos()
    E = rows * cols
    y = np.zeros(E)
    for e in range(E):
        a = None
        for r, (cc, ss, z, sts) in enumerate(shards):
            code = Fraction(float(table[cc[e]]))
            sc = Fraction(float(np.float32(sts[0]) * table[ss[e // B]]))
            a = _round_f32(code * sc) if r == 0 else _round_f32(code * sc + Fraction(a))
        y[e] = a
    y = y.astype(np.float32).reshape(-1, B)
    a_b = np.abs(y).max(axis=1).astype(np.float64)
    if mode == 1:
        assert st[1] == np.float32(a_b.max()) and st[0] == orc.scale_from_amax(st[1])
    S = float(st[0])
    ok = _nearest_codes(a_b / (448.0 * S), table)[np.arange(len(a_b)), s]
    assert np.all(ok | ((s == 1) & (a_b > 0)))
    sb = (np.float32(S) * table[s]).astype(np.float64)
    for b in range(len(a_b)):
        near = _nearest_codes(np.clip(y[b] / sb[b], -448, 448), table)
        assert np.all(near[np.arange(B), c.reshape(-1, B)[b]])
    # round trip to the original domain against the float64 sum of the inputs
    out = orc.decompress(0, B, c, s, None, st, 1, rows, cols, orc.FP32).astype(np.float64)
    ref = np.stack(deq).astype(np.float64).sum(axis=0)
    err = np.sqrt(((out - ref) ** 2).reshape(-1, B).sum(axis=1))
    bound = np.sqrt((np.abs(y).astype(np.float64) ** 2).sum(axis=1)) / np.sqrt(B) * (2.0 ** -4 + 1e-5) \
        + n * 1e-6 * np.abs(ref).reshape(-1, B).max(axis=1) * np.sqrt(B)
    assert np.all(err <= bound)
