"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
binding and the CPU oracle on the same bytes, and compare."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as orc
import quantized_tensor_activation_gb300 as qta

DT_TORCH = {qta.BF16: torch.bfloat16, qta.FP16: torch.float16, qta.FP32: torch.float32}
ORC_DT = {qta.BF16: orc.BF16, qta.FP16: orc.FP16, qta.FP32: orc.FP32}
ORC_SCH = {qta.TACO_FP8: orc.TACO_FP8, qta.INT8_SYM_B64: orc.INT8_SYM, qta.INT4_ASYM_G128: orc.INT4_ASYM,
           qta.INT8_ASYM_G128: orc.INT8_ASYM}
BLOCK_OF = {qta.INT8_SYM_B64: 64, qta.INT4_ASYM_G128: 128, qta.INT8_ASYM_G128: 128}

# The floating-point tolerance of the FP32 outputs (reduce sums, fp32
# decompression): max relative error 1e-5; the kernels replicate the oracle's
# operation order, so equality is expected and counted as well.
REL_TOL = 1e-5


def device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw bytes of a tensor as a flat numpy array of the matching uint type."""
    t = t.detach().cpu().contiguous()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16).reshape(-1)
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy().view(np.uint32).reshape(-1)
    if t.dtype == torch.int8:
        return t.numpy().view(np.uint8).reshape(-1)
    return t.numpy().reshape(-1)


def host_bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a).reshape(-1)
    if a.dtype == np.float32:
        return a.view(np.uint32)
    if a.dtype == np.int8:
        return a.view(np.uint8)
    return a


def assert_same(name: str, gpu, ref) -> None:
    g = bits(gpu) if isinstance(gpu, torch.Tensor) else host_bits(gpu)
    r = host_bits(ref)
    if g.dtype != r.dtype:
        g = g.view(r.dtype)
    assert g.size == r.size, f"{name}: size {g.size} != {r.size}"
    bad = np.flatnonzero(g != r)
    assert bad.size == 0, f"{name}: {bad.size} of {r.size} differ, first at {bad[:8].tolist()}: " \
                          f"gpu {g[bad[:4]].tolist()} oracle {r[bad[:4]].tolist()}"


def assert_close_f32(name: str, gpu: torch.Tensor, ref: np.ndarray) -> None:
    g = gpu.detach().cpu().numpy().reshape(-1).astype(np.float64)
    r = np.asarray(ref, dtype=np.float32).reshape(-1).astype(np.float64)
    err = np.abs(g - r)
    ok = err <= REL_TOL * np.abs(r) + 1e-37
    assert ok.all(), f"{name}: {int((~ok).sum())} of {r.size} beyond rel {REL_TOL}, max err {err.max()}"


def random_values(rng, shape, kind="mixed", scale=1.0):
    if kind == "mixed":
        x = rng.standard_normal(shape) * 0.02
        out = rng.random(shape) < 0.02
        x = np.where(out, rng.standard_normal(shape), x)
        ch = rng.choice(shape[-1], max(1, shape[-1] // 100), replace=False)
        x[..., ch] *= 10
    elif kind == "laplace":
        x = rng.laplace(0, 0.01, shape)
    elif kind == "t":
        x = rng.standard_t(3, shape) * 0.05
    else:
        x = rng.standard_normal(shape)
    return (x * scale).astype(np.float32)


def to_dtype_cpu(x: np.ndarray, dtype: int) -> torch.Tensor:
    return torch.from_numpy(x).to(DT_TORCH[dtype])


def oracle_bits_in(xt: torch.Tensor) -> np.ndarray:
    """Input bytes for the oracle, exactly those handed to the GPU."""
    return bits(xt) if xt.dtype != torch.float32 else xt.numpy().reshape(-1)


def gpu_compress(scheme, B, xt: torch.Tensor, dtype, batch, rows, cols, mode=qta.SCALE_CURRENT, state=None,
                 dev=None):
    d = qta.desc(scheme, B, rows, cols, batch=batch)
    q = qta.alloc_qtensor(d, dev)
    if state is not None and q.state is not None:
        q.state.copy_(torch.from_numpy(state))
    qta.taco_compress(d, xt.to(dev), dtype, q, mode)
    return d, q


def oracle_compress(scheme, B, xt, dtype, batch, rows, cols, mode=orc.CURRENT, state=None):
    st = None
    if scheme == qta.TACO_FP8:
        st = np.zeros(2 * batch, dtype=np.float32) if state is None else state.copy()
    c, s, z = orc.compress(ORC_SCH[scheme], B, oracle_bits_in(xt), ORC_DT[dtype], batch, rows, cols, st, mode)
    return c, s, z, st


def compare_qtensor(name, q, ref):
    c, s, z, st = ref
    assert_same(name + " codes", q.codes, c)
    assert_same(name + " scales", q.scales, s)
    if z is not None:
        assert_same(name + " zeros", q.zeros, z)
    if st is not None:
        assert_same(name + " state", q.state, st)
