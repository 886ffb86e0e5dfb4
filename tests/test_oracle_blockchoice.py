"""Pins of the per-tensor block-size choice (TACO's data-driven reshape read
as: the candidate block size with the smallest round-trip error)."""
import numpy as np
import pytest
import scipy.linalg


def _exact_for(B, nblocks, rng):
    """x = H_B c / B per block, c integers in [-16, 16] with one +-448 per
    block: with block size B the transform is c itself, every block scale is
    1 and the round trip is exact."""
    c = rng.integers(-16, 17, size=(nblocks, B)).astype(np.float64)
    c[np.arange(nblocks), rng.integers(0, B, nblocks)] = 448.0 * rng.choice([-1, 1], nblocks)
    x = c @ scipy.linalg.hadamard(B).T / B
    return x.reshape(-1).astype(np.float32)


@pytest.mark.parametrize("B", [64, 128, 256])
def test_exactly_representable_block_size_is_chosen(orc, B):
    rng = np.random.default_rng(B)
    rows, cols = 4, 1024
    x = _exact_for(B, rows * cols // B, rng)
    best, errs = orc.choose_block(x, orc.FP32, 1, rows, cols)
    assert best == B and errs[B] == 0.0
    assert all(e > 0 for b, e in errs.items() if b != B)


def test_ties_and_candidates(orc):
    x = np.zeros(2 * 512, dtype=np.float32)
    best, errs = orc.choose_block(x, orc.FP32, 1, 2, 512)
    assert best == 64 and set(errs) == {64, 128, 256} and all(e == 0 for e in errs.values())
    _, errs = orc.choose_block(np.zeros(192, np.float32), orc.FP32, 1, 1, 192)
    assert set(errs) == {64}                               # 128, 256 do not divide 192


def test_outlier_channels_prefer_larger_blocks(orc):
    # one dominant channel per 256 columns: a wider rotation spreads it over
    # more elements, so the round-trip error falls with B
    rng = np.random.default_rng(1)
    rows, cols = 64, 1024
    x = rng.standard_normal((rows, cols)).astype(np.float32) * 0.01
    x[:, ::256] *= 3000.0
    _, errs = orc.choose_block(x.reshape(-1), orc.FP32, 1, rows, cols)
    assert errs[256] < errs[128] < errs[64]
