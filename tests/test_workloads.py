"""The seeded input generators produce finite values of the stated shapes
(no CUDA, no codec arithmetic)."""
import math

import torch

import workloads as W


def test_laplace_endpoints_are_finite():
    r = torch.tensor([0.0, 0.5 - 2.0 ** -24, 0.5, 1.0 - 2.0 ** -24], dtype=torch.float32)
    x = W.laplace_from_uniform(r, 0.01)
    assert torch.isfinite(x).all()
    # the extreme cells sit at -/+ b ln(2^24), the middle ones next to 0
    assert math.isclose(float(x[0]), -0.01 * 24 * math.log(2), rel_tol=1e-6)
    assert math.isclose(float(x[3]), 0.01 * 24 * math.log(2), rel_tol=1e-6)
    assert abs(float(x[1])) < 1e-8 and abs(float(x[2])) < 1e-8 and float(x[1]) < 0 < float(x[2])


def test_laplace_moments():
    g = torch.Generator().manual_seed(3)
    x = W.laplace_from_uniform(torch.rand(1 << 20, generator=g), 0.01).double()
    assert abs(float(x.mean())) < 1e-4
    assert math.isclose(float(x.abs().mean()), 0.01, rel_tol=0.01)      # E|x| = b


def test_every_workload_is_finite_and_shaped():
    for name, w in W.WORKLOADS.items():
        x = W.make_rank_inputs(w, rows=64, ranks=2)
        assert x.shape == (2, 64, w.cols) and x.dtype == w.torch_dtype, name
        assert torch.isfinite(x.float()).all(), name
        ch = W.outlier_channels(w)
        assert ch.unique().numel() == ch.numel() and (ch < w.cols).all(), name
