"""Pins of the oracle's block Hadamard (the rotation of TACO's Adaptive
Scale-Hadamard transform; TACO Core claim, Fig. 7, Fig. 8).

* The transform of each unit vector e_k is column k of scipy's Sylvester
  Hadamard matrix, exactly; H H^T = B I in integers.
* On small-integer inputs the FP32 butterfly is exact, so it equals the
  integer product H x computed in int64.
* On real inputs it agrees with the float64 dense product within the
  butterfly's rounding bound, and the inverse (same butterfly, times 1/B)
  recovers the input within 2 log2(B) ulps of the block's scale.
"""
import numpy as np
import pytest
import scipy.linalg


@pytest.mark.parametrize("B", [2, 4, 8, 16, 32, 64, 128, 256])
def test_unit_vectors_give_hadamard_columns(orc, B):
    eye = np.eye(B, dtype=np.float32)
    cols = orc.fwht(eye.reshape(-1), B).reshape(B, B)   # row k = transform of e_k
    H = scipy.linalg.hadamard(B)
    assert np.array_equal(cols.T.astype(np.int64), H)
    Hi = cols.astype(np.int64)
    assert np.array_equal(Hi @ Hi.T, B * np.eye(B, dtype=np.int64))
    # Sylvester entry rule (-1)^popcount(i & j)
    i, j = np.meshgrid(np.arange(B), np.arange(B), indexing="ij")
    pc = np.vectorize(lambda v: bin(int(v)).count("1"))(i & j)
    assert np.array_equal(H, np.where(pc % 2 == 0, 1, -1))


@pytest.mark.parametrize("B", [64, 128, 256])
def test_integer_inputs_exact(orc, B):
    rng = np.random.default_rng(B)
    x = rng.integers(-1000, 1001, size=(50, B)).astype(np.int64)
    y = orc.fwht(x.astype(np.float32).reshape(-1), B).reshape(50, B)
    ref = x @ scipy.linalg.hadamard(B).T
    assert np.array_equal(y.astype(np.int64), ref)


@pytest.mark.parametrize("B", [64, 128, 256])
def test_float_inputs_within_rounding_bound(orc, B):
    rng = np.random.default_rng(10 + B)
    x = (rng.standard_normal((200, B)) * np.exp(rng.uniform(-8, 8, (200, 1)))).astype(np.float32)
    y = orc.fwht(x.reshape(-1), B).reshape(200, B).astype(np.float64)
    ref = x.astype(np.float64) @ scipy.linalg.hadamard(B).T.astype(np.float64)
    # each output is a sum of B terms formed by a depth-log2(B) adder tree
    eps = 2.0 ** -24
    bound = np.log2(B) * eps * np.abs(x).astype(np.float64).sum(axis=1, keepdims=True) * 1.01
    assert np.all(np.abs(y - ref) <= bound)
    # inverse: same butterfly then 1/B recovers x
    back = orc.fwht(y.astype(np.float32).reshape(-1), B).reshape(200, B) * np.float32(1.0 / B)
    err = np.abs(back.astype(np.float64) - x)
    assert np.all(err <= 2 * np.log2(B) * eps * np.abs(x).max(axis=1, keepdims=True) * np.sqrt(B))


def test_butterfly_order_is_ascending(orc):
    # A value pattern whose FP32 result depends on the summation order: the
    # ascending-stride butterfly adds neighbours first.  For x = (1, 2^-24, -1,
    # 0...) with B = 4: stage h=1 gives (1+2^-24 -> 1, ...), stage h=2 then
    # cancels to exactly 0 in output 0; a descending order would keep 2^-24.
    x = np.array([1.0, 2.0 ** -24, -1.0, 0.0], dtype=np.float32)
    y = orc.fwht(x, 4)
    assert y[0] == 0.0
