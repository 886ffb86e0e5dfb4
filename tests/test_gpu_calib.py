"""GPU: the squared-error reduction and the per-tensor block-size choice
against numpy and the oracle."""
import numpy as np
import pytest
import torch

import oracle as orc
import quantized_tensor_activation_gb300 as qta
from quantized_tensor_activation_gb300 import calib
from gpu_util import ORC_DT, device, oracle_bits_in, random_values, to_dtype_cpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [qta.BF16, qta.FP16, qta.FP32])
@pytest.mark.parametrize("n", [1, 255, 4096 + 17, 3 << 20])
def test_sq_error(dtype, n):
    dev = device()
    rng = np.random.default_rng(n + dtype)
    a = to_dtype_cpu(random_values(rng, (n,), "mixed"), dtype)
    b = torch.from_numpy(random_values(rng, (n,), "mixed"))
    out = torch.full((1,), 123.0, dtype=torch.float64, device=dev)
    qta.qta_sq_error(a.to(dev), dtype, b.to(dev), n, out)
    want = float(((a.double() - b.double()) ** 2).sum())
    assert abs(out.item() - want) <= 1e-12 * want + 1e-300


def test_sq_error_empty():
    dev = device()
    out = torch.full((1,), 5.0, dtype=torch.float64, device=dev)
    qta.qta_sq_error(None, qta.BF16, None, 0, out)
    assert out.item() == 0.0


@pytest.mark.parametrize("B", [64, 128, 256])
def test_exact_block_size_is_chosen(B):
    dev = device()
    import scipy.linalg
    rng = np.random.default_rng(B)
    rows, cols = 8, 1024
    nb = rows * cols // B
    c = rng.integers(-16, 17, size=(nb, B)).astype(np.float64)
    c[np.arange(nb), rng.integers(0, B, nb)] = 448.0
    x = torch.from_numpy((c @ scipy.linalg.hadamard(B).T / B).astype(np.float32).reshape(rows, cols))
    best, errs = calib.choose_block(x.to(dev))
    assert best == B and errs[B] == 0.0


@pytest.mark.parametrize("dtype", [qta.BF16, qta.FP16])
def test_block_errors_match_oracle(dtype):
    dev = device()
    rng = np.random.default_rng(3 + dtype)
    batch, rows, cols = 2, 48, 1024
    xv = random_values(rng, (batch, rows, cols), "mixed")
    xv[..., ::256] *= 40.0
    xt = to_dtype_cpu(xv, dtype)
    best, errs = calib.choose_block(xt.to(dev))
    obest, oerrs = orc.choose_block(oracle_bits_in(xt), ORC_DT[dtype], batch, rows, cols)
    assert set(errs) == set(oerrs)
    for b in errs:
        assert abs(errs[b] - oerrs[b]) <= 1e-9 * oerrs[b]
    assert best == obest
