"""Exact pins of the oracle's integer schemes (EQuARX block-symmetric INT8,
Flash Communication asymmetric group-128 INT4 / INT8).

What is pinned, and by what:
  * the tie rule (every rounding is round-to-nearest-even, a reading: the
    pages state none): inputs built so that the scaled value is exactly
    k + 1/2, with power-of-two scales and exactly representable inputs, so the
    only correct code is the even neighbour -- a half-away-from-zero or
    half-up rounding gives the odd one;
  * the stored FP32 scale of INT8 (EQuARX: one FP32 scale per 64 entries):
    bit-equal to the correctly rounded a/127 (a two-rounding a * (1/127)
    differs on the same data, which the test checks, so it has power);
  * the codes and metadata of both schemes on random data: equal to the
    reading's operations evaluated in exact rational arithmetic with one
    IEEE rounding per operation (tests/exact_round.py), not by the float unit;
  * the asymmetric reduce (Flash Communication: local FP32 sum of the
    dequantized shards): acc = RN(q0 s0 + z0), then acc = RN(acc + RN(q s + z))
    per rank in rank order, in exact arithmetic; a fused fmaf(q, s, acc + z)
    or a single rounding of the whole term differs on the same data.
"""
from fractions import Fraction

import numpy as np
import pytest

from exact_round import fr, rf16, rf32, rint_even


def _f16val(bits):
    return fr(np.uint16(bits).view(np.float16))


# ------------------------------------------------------------------ INT8 sym
@pytest.mark.parametrize("in_dtype", ["fp32", "bf16"])
def test_int8_sym_ties_go_to_even(orc, in_dtype):
    # block 0: absmax 127 -> inv = 127/127 = 1, x = k + 1/2 scales to k + 1/2
    # block 1: absmax 254 -> inv = 127/254 = 1/2 exactly, x = 2k + 1 scales to k + 1/2
    k = np.array([0, 1, 2, 3, 10, 125, -1, -2, -3, -126, 62, 63, 64, 99, 100, -100], dtype=np.float64)
    b0 = np.concatenate([k + 0.5, [127.0]])
    b1 = np.concatenate([2 * k + 1, [254.0]])
    blocks = []
    for b in (b0, b1):
        x = np.zeros(64)
        x[:b.size] = b
        blocks.append(x)
    x = np.concatenate(blocks).astype(np.float32)
    if in_dtype == "bf16":
        xb = orc.f32_to_bf16(x)
        assert np.array_equal(orc.bf16_to_f32(xb), x)          # every value is exact in bf16
        codes, scales, _ = orc.compress(orc.INT8_SYM, 64, xb, orc.BF16, 1, 2, 64)
    else:
        codes, scales, _ = orc.compress(orc.INT8_SYM, 64, x, orc.FP32, 1, 2, 64)
    assert scales[0] == np.float32(1.0) and scales[1] == np.float32(2.0)
    want = np.array([rint_even(Fraction(2 * int(kk) + 1, 2)) for kk in k])
    for blk in range(2):
        got = codes[blk * 64: blk * 64 + k.size].astype(np.int64)
        assert np.array_equal(got, want), (blk, got, want)
        assert np.all(got % 2 == 0)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("zero", [0.0, -1.0, 3.5])
def test_asym_ties_go_to_even(orc, bits, zero):
    # group min z, step s = 2^-3 (INT8) or 2^-2 (INT4), group max z + Q s: then
    # (max - min) / Q = s and 1/s are exact, and x = z + (k + 1/2) s scales to
    # exactly k + 1/2; the correct code is the even one of k, k + 1.
    Q = 2 ** bits - 1
    s = 0.125 if bits == 8 else 0.25
    scheme = orc.INT8_ASYM if bits == 8 else orc.INT4_ASYM
    ks = np.arange(Q)                                          # k + 1/2 for k = 0 .. Q-1
    x = np.empty(128)
    x[0], x[1] = zero, zero + Q * s
    rest = zero + (np.resize(ks, 126) + 0.5) * s
    x[2:] = rest
    x = x.astype(np.float32)
    assert np.all(x.astype(np.float64) == np.concatenate([[zero, zero + Q * s], rest]))
    codes, scales, zeros = orc.compress(scheme, 128, x, orc.FP32, 1, 1, 128)
    assert _f16val(scales[0]) == Fraction(s) and _f16val(zeros[0]) == Fraction(zero)
    q = codes if bits == 8 else np.stack([codes & 15, codes >> 4], axis=1).reshape(-1)
    q = q.astype(np.int64)
    assert q[0] == 0 and q[1] == Q
    want = np.array([rint_even(Fraction(2 * int(k) + 1, 2)) for k in np.resize(ks, 126)])
    assert np.array_equal(q[2:], want)
    assert np.all(q[2:] % 2 == 0)


def test_int8_sym_scale_is_correctly_rounded(orc):
    rng = np.random.default_rng(17)
    nb = 400
    x = (rng.standard_normal((nb, 64)) * np.exp(rng.uniform(-6, 6, (nb, 1)))).astype(np.float32)
    x[7] = 0
    codes, scales, _ = orc.compress(orc.INT8_SYM, 64, x.reshape(-1), orc.FP32, 1, nb, 64)
    a = [fr(v) for v in np.abs(x).max(axis=1)]
    want = np.array([float(rf32(ai / 127)) for ai in a], dtype=np.float32)
    assert np.array_equal(scales.view(np.uint32), want.view(np.uint32))
    # the same data tells a two-rounding a * RN(1/127) apart
    r127 = rf32(Fraction(1, 127))
    alt = np.array([float(rf32(ai * r127)) for ai in a], dtype=np.float32)
    assert np.any(alt.view(np.uint32) != want.view(np.uint32))


def test_int8_sym_codes_exact(orc):
    # q = clamp(rint(RN(x * RN(127 / a))), -127, 127), every operation once
    # rounded, evaluated exactly
    rng = np.random.default_rng(23)
    nb = 48
    x = (rng.standard_normal((nb, 64)) * np.exp(rng.uniform(-4, 4, (nb, 1)))).astype(np.float32)
    x[5] = 0
    codes, _, _ = orc.compress(orc.INT8_SYM, 64, x.reshape(-1), orc.FP32, 1, nb, 64)
    c = codes.reshape(nb, 64).astype(np.int64)
    for b in range(nb):
        a = max(abs(fr(v)) for v in x[b])
        if a == 0:
            assert np.all(c[b] == 0)
            continue
        inv = rf32(Fraction(127) / a)
        for i in range(64):
            q = max(-127, min(127, rint_even(rf32(fr(x[b, i]) * inv))))
            assert c[b, i] == q, (b, i)


# ------------------------------------------------------------------ ASYM
def _asym_ref(xg, bits):
    """Scale, zero and codes of one group by the reading, exactly."""
    Q = 2 ** bits - 1
    xs = [fr(v) for v in xg]
    mn, mx = min(xs), max(xs)
    sf = rf32(rf32(mx - mn) / Q)
    sf = min(sf, Fraction(65504))
    zc = max(min(mn, Fraction(65504)), Fraction(-65504))
    s = rf16(sf)
    z = rf16(zc)
    inv = rf32(1 / s) if s > 0 else Fraction(0)
    q = [max(0, min(Q, rint_even(rf32(rf32(v - z) * inv)))) for v in xs]
    return s, z, q


@pytest.mark.parametrize("bits", [4, 8])
def test_asym_codes_exact(orc, bits):
    scheme = orc.INT4_ASYM if bits == 4 else orc.INT8_ASYM
    rng = np.random.default_rng(31 + bits)
    ng = 24
    x = (rng.standard_t(3, size=(ng, 128)) * np.exp(rng.uniform(-5, 3, (ng, 1)))).astype(np.float32)
    x[3] = 0.75
    codes, scales, zeros = orc.compress(scheme, 128, x.reshape(-1), orc.FP32, 1, ng, 128)
    q = codes if bits == 8 else np.stack([codes & 15, codes >> 4], axis=1).reshape(-1)
    q = q.reshape(ng, 128).astype(np.int64)
    for g in range(ng):
        s, z, qr = _asym_ref(x[g], bits)
        assert _f16val(scales[g]) == s and _f16val(zeros[g]) == z, g
        assert np.array_equal(q[g], np.array(qr)), g


# ------------------------------------------------------------------ reduce
def _dequant_terms(orc, shards, bits, e):
    """(q, s, z) of element e of every rank, exactly."""
    out = []
    for c, s, z, _ in shards:
        if bits == 8:
            q = int(c[e])
        else:
            q = int((c[e >> 1] >> ((e & 1) * 4)) & 15)
        out.append((Fraction(q), _f16val(s[e // 128]), _f16val(z[e // 128])))
    return out


@pytest.mark.parametrize("bits", [4, 8])
def test_reduce_asym_one_rounding_per_term(orc, bits):
    scheme = orc.INT4_ASYM if bits == 4 else orc.INT8_ASYM
    rng = np.random.default_rng(40 + bits)
    rows, cols, n = 2, 256, 4
    shards = []
    for r in range(n):
        # odd groups: Student-t values (there q s + z is mostly exact and the
        # orders agree); even groups: positive values with a tiny minimum
        # (z's last bit far below s), where q s + z needs more than 24 bits and
        # the order of the roundings shows
        x = rng.standard_t(3, size=(rows, cols)) * (0.05 * (1 + r))
        g = x.reshape(-1, 128)
        g[0::2] = rng.uniform(0, 8.0 * (1 + r), size=g[0::2].shape)
        g[0::2, 5] = rng.uniform(1e-4, 3e-4, size=g[0::2, 5].shape)
        x = g.astype(np.float32).reshape(-1)
        c, s, z = orc.compress(scheme, 128, x, orc.FP32, 1, rows, cols)
        shards.append((c, s, z, None))
    out = orc.reduce(scheme, 128, shards, rows, cols)
    E = rows * cols
    want = np.zeros(E, dtype=np.float32)
    alt_fused = np.zeros(E, dtype=np.float32)      # acc = RN(q s + RN(acc + z))
    alt_one = np.zeros(E, dtype=np.float32)        # acc = RN(acc + q s + z)
    for e in range(E):
        terms = _dequant_terms(orc, shards, bits, e)
        a = b = c1 = None
        for r, (q, s, z) in enumerate(terms):
            d = rf32(q * s + z)
            if r == 0:
                a = b = c1 = d
            else:
                a = rf32(a + d)
                b = rf32(q * s + rf32(b + z))
                c1 = rf32(c1 + q * s + z)
        want[e], alt_fused[e], alt_one[e] = float(a), float(b), float(c1)
    assert np.array_equal(out.view(np.uint32), want.view(np.uint32))
    assert np.any(alt_fused.view(np.uint32) != want.view(np.uint32))
    assert np.any(alt_one.view(np.uint32) != want.view(np.uint32))


# ------------------------------------------------------------------ TACO
def _e4m3_values():
    import torch
    t = torch.arange(0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    return [fr(v) for v in t]                       # codes 0x00 .. 0x7E, ascending


def _enc8(v, table):
    """E4M3 code of an exact value: nearest of the 127 magnitudes, ties to the
    even code, magnitudes above 448 saturate; the sign bit is kept."""
    a = abs(v)
    if a > table[-1]:
        c = 0x7E
    else:
        c = min(range(len(table)), key=lambda i: (abs(table[i] - a), i % 2))
    return c | (0x80 if v < 0 else 0)


# S = 7.3: a block with a_b = 1 whose scale byte rounds to 0 and takes the
# 2^-9 floor.  S = 0.0018796994 (binary32): for a_b = 1 the ratio RN(1/RN(448 S))
# is 1.1874999 (byte 0x39), while (1/448)/S rounded twice gives the tie 1.1875
# (byte 0x3A) -- the two forms of the factor are told apart.
@pytest.mark.parametrize("S_value", [7.3, 0.0018796994])
@pytest.mark.parametrize("B", [64, 128])
def test_taco_scale_bytes_and_codes_exact(orc, B, S_value):
    # Small-integer blocks, so the FP32 butterfly is exact and y = H x is known
    # in integers; a stale per-tensor scale S (DELAYED).  Reading: t =
    # RN(1 / RN(448 S)), r_b = E4M3(RN(a_b t)) (2^-9 when that is 0 while
    # a_b > 0), s_b = RN(S r_b), inv = RN(1 / s_b), q = E4M3_sat(RN(y inv)).
    import scipy.linalg
    rng = np.random.default_rng(70 + B)
    nb = 20
    xi = rng.integers(-60, 61, size=(nb, B))
    xi[::4] *= 7
    xi[2] = 0
    xi[5] = 0
    xi[5, 3] = 1                                    # a_b = 1: the ratio rounds to 0 -> r_b = 2^-9
    xi[6] = 0
    xi[6, :2] = 3                                   # a_b = 6
    S = np.float32(S_value)
    st = np.array([S, 0.0], dtype=np.float32)
    codes, scales, _ = orc.compress(orc.TACO_FP8, B, xi.astype(np.float32).reshape(-1), orc.FP32, 1, nb, B,
                                    st, orc.DELAYED)
    y = xi @ scipy.linalg.hadamard(B).T
    table = _e4m3_values()
    Sf = fr(S)
    t = rf32(1 / rf32(448 * Sf))
    c = codes.reshape(nb, B)
    if S_value == 7.3:
        assert scales[5] == 0x01
    else:
        assert rf32(rf32(Fraction(1) / 448) / Sf) == Fraction(19, 16) and _enc8(t, table) == 0x39
        assert scales[5] == 0x39
    for b in range(nb):
        a = Fraction(int(np.abs(y[b]).max()))
        r = _enc8(rf32(a * t), table)
        if r == 0 and a > 0:
            r = 0x01
        assert scales[b] == r, b
        sb = rf32(Sf * table[r])
        inv = rf32(1 / sb) if sb > 0 else Fraction(0)
        for i in range(B):
            assert c[b, i] == _enc8(rf32(Fraction(int(y[b, i])) * inv), table), (b, i)
    assert st[1] == np.float32(np.abs(y).max())
