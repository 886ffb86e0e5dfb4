"""Failure detection on the GPU without a fault: a bounded pipeline wait that
nothing completes runs out, the kernel records the timeout and returns, the
host reads the flag, and the context keeps working."""
import time

import numpy as np
import pytest
import torch

import oracle as orc
import quantized_tensor_activation_gb300 as qta
from gpu_util import compare_qtensor, device, gpu_compress, oracle_compress, random_values, to_dtype_cpu

pytestmark = pytest.mark.gpu


def test_wait_expiry_is_reported_and_the_context_survives():
    dev = device()
    qta.qta_device_error(True)
    qta.qta_wait_self_test(True)                     # the barrier completes: no flag
    assert qta.qta_device_error() == 0
    t0 = time.perf_counter()
    qta.qta_wait_self_test(False)                    # nothing arrives: the wait runs out
    flags = qta.qta_device_error()
    dt = time.perf_counter() - t0
    assert flags & 1, flags
    assert 1.5 < dt < 60, dt
    assert qta.qta_device_error() == 0               # reading cleared it
    # the same context still computes correctly
    rng = np.random.default_rng(0)
    xt = to_dtype_cpu(random_values(rng, (2, 16, 512), "mixed"), qta.BF16)
    _, q = gpu_compress(qta.TACO_FP8, 128, xt, qta.BF16, 2, 16, 512, qta.SCALE_CURRENT, dev=dev)
    torch.cuda.synchronize()
    compare_qtensor("after timeout", q, oracle_compress(qta.TACO_FP8, 128, xt, qta.BF16, 2, 16, 512, orc.CURRENT))
    assert qta.qta_device_error() == 0
