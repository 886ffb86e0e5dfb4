"""Pins of the oracle's number formats against things other than itself.

* E4M3 decode against torch's float8_e4m3fn (a library routine) on all codes.
* E4M3 encode over all 2^32 binary32 patterns: against an independent
  nearest-value table search for every pattern whose magnitude lies in
  [2^-12, 2^10); against the constant each remaining pattern must give
  (signed zero below, +-448 above and for +-Inf, 0x7F for NaN); on random
  patterns; against torch's RNE cast in range.
* TACO Fig. 6, Eq. (3): |x - FP8(x)| <= 2^(floor(log2|x|) - m), m = 3.
* bf16 / fp16 rounding against torch's casts (round-to-nearest-even).
"""
import numpy as np
import pytest
import torch


def _torch_e4m3_table():
    codes = torch.arange(256, dtype=torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float32).numpy()


def test_e4m3_decode_matches_torch_all_codes(orc):
    mine = orc.e4m3_decode(np.arange(256))
    ref = _torch_e4m3_table()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(mine[~nan].view(np.uint32), ref[~nan].view(np.uint32))  # incl. -0
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9 and mine[0x08] == 2.0 ** -6


def test_e4m3_roundtrip_every_code(orc):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(orc.e4m3_encode(orc.e4m3_decode(codes)), codes)


def _table_search_encode(v: np.ndarray) -> np.ndarray:
    """Independent encoder: nearest finite E4M3 value by search, ties to the
    even code, magnitudes past 448 saturate; NaN -> 0x7F; sign kept."""
    table = _torch_e4m3_table()
    pos = table[:0x7F].astype(np.float64)          # codes 0x00..0x7E ascending
    a = np.abs(v.astype(np.float64))
    idx = np.searchsorted(pos, a)                   # pos[idx-1] < a <= pos[idx]
    hi = np.clip(idx, 0, 0x7E)
    lo = np.clip(idx - 1, 0, 0x7E)
    dlo = a - pos[lo]
    dhi = pos[hi] - a
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    # beyond 448: above the (virtual) midpoint 464 it saturates too
    pick = np.where(a > 448.0, 0x7E, pick).astype(np.uint8)
    sign = (np.signbit(v).astype(np.uint8) << 7)
    out = pick | sign
    return np.where(np.isnan(v), np.uint8(0x7F), out).astype(np.uint8)


def test_e4m3_encode_exhaustive_band(orc):
    # every binary32 pattern with biased exponent 115..136 (|v| in [2^-12, 2^10)),
    # both signs: 22 * 2^23 * 2 = 369M values, checked in chunks
    lo = 115 << 23
    hi = 137 << 23
    step = 1 << 22
    for start in range(lo, hi, step):
        u = np.arange(start, min(start + step, hi), dtype=np.uint32)
        for sgn in (0, 0x80000000):
            v = (u | np.uint32(sgn)).view(np.float32)
            assert np.array_equal(orc.e4m3_encode(v), _table_search_encode(v)), hex(start)


def test_e4m3_encode_every_pattern_outside_the_band(orc):
    # the remaining binary32 patterns, every one: below the band (|v| < 2^-12,
    # under a quarter of the smallest subnormal step) the code is a signed zero;
    # above it (|v| >= 2^10 > 464, and +-Inf) the code saturates to +-448; NaN
    # gives 0x7F.  With the band test this covers all 2^32 patterns.
    step = 1 << 24
    for lo, hi, pos_code, neg_code in ((0, 115 << 23, 0x00, 0x80), (137 << 23, 255 << 23, 0x7E, 0xFE),
                                       (255 << 23, (255 << 23) + 1, 0x7E, 0xFE)):
        for start in range(lo, hi, step):
            u = np.arange(start, min(start + step, hi), dtype=np.uint32)
            for sgn, code in ((0, pos_code), (0x80000000, neg_code)):
                got = orc.e4m3_encode((u | np.uint32(sgn)).view(np.float32))
                assert np.all(got == code), hex(start)
    nan = np.arange((255 << 23) + 1, 1 << 31, dtype=np.uint32)
    for sgn in (0, 0x80000000):
        assert np.all(orc.e4m3_encode((nan | np.uint32(sgn)).view(np.float32)) == 0x7F)


def test_e4m3_encode_random_patterns(orc):
    rng = np.random.default_rng(1)
    u = rng.integers(0, 2 ** 32, size=4_000_000, dtype=np.uint64).astype(np.uint32)
    v = u.view(np.float32)
    mine = orc.e4m3_encode(v)
    ref = _table_search_encode(v)
    assert np.array_equal(mine, ref)
    specials = np.array([np.inf, -np.inf, 0.0, -0.0, 464.0, 464.0001, 463.99997, 1e30,
                         2 ** -10, 2 ** -10 * 1.0000001, 3 * 2 ** -10, -(2 ** -126)], dtype=np.float32)
    assert list(orc.e4m3_encode(specials)) == [0x7E, 0xFE, 0x00, 0x80, 0x7E, 0x7E, 0x7E, 0x7E,
                                                 0x00, 0x01, 0x02, 0x80]


def test_e4m3_encode_matches_torch_in_range(orc):
    rng = np.random.default_rng(2)
    v = np.concatenate([
        rng.standard_normal(1_000_000).astype(np.float32) * 50,
        rng.uniform(-464, 464, 1_000_000).astype(np.float32),
        # all midpoints between neighbouring finite codes (ties)
        ((_torch_e4m3_table()[:0x7E] + _torch_e4m3_table()[1:0x7F]) / 2).astype(np.float32),
    ])
    v = v[np.abs(v) <= 464]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(orc.e4m3_encode(v), ref)


def test_eq3_ulp_bound(orc):
    # TACO Fig. 6, Eq. (3): in-range error bounded by one ULP 2^(floor(log2|x|)-m),
    # m = 3 mantissa bits; round-to-nearest gives half of it.
    rng = np.random.default_rng(3)
    v = np.exp2(rng.uniform(-6, np.log2(448), 2_000_000)).astype(np.float32)
    v *= np.where(rng.random(v.size) < 0.5, -1, 1).astype(np.float32)
    q = orc.e4m3_decode(orc.e4m3_encode(v)).astype(np.float64)
    e = np.abs(v.astype(np.float64) - q)
    ulp = np.exp2(np.floor(np.log2(np.abs(v.astype(np.float64)))) - 3)
    assert np.all(e <= ulp)
    assert np.all(e <= ulp / 2)


def test_bf16_fp16_rounding_matches_torch(orc):
    rng = np.random.default_rng(4)
    u = rng.integers(0, 2 ** 32, size=3_000_000, dtype=np.uint64).astype(np.uint32)
    v = u.view(np.float32)
    v = v[~np.isnan(v)]
    extra = np.array([65504, 65519.99, 65520, 65536, 2 ** -24, 2 ** -25, 3 * 2 ** -26,
                      2 ** -25 * 1.0000001, -0.0, np.inf, 3.3895314e38, 3.4e38], dtype=np.float32)
    near = (rng.standard_normal(2_000_000) * 100).astype(np.float32)
    v = np.concatenate([v, extra, near])
    bf = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    hf = torch.from_numpy(v).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.f32_to_bf16(v), bf)
    assert np.array_equal(orc.f32_to_f16(v), hf)
    h = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(h.view(np.int16)).view(torch.float16).to(torch.float32).numpy()
    mine = orc.f16_to_f32(h)
    fin = ~np.isnan(ref)
    assert np.array_equal(np.isnan(mine), ~fin)
    assert np.array_equal(mine[fin].view(np.uint32), ref[fin].view(np.uint32))
