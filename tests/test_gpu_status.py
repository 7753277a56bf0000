"""Failure reporting on the GPU, made without a fault.

The library's self-test launches one wait on an mbarrier that nothing completes, with a 20 ms
limit -- the bounded wait every pipeline of the library goes through.  The wait gives up and
records TE_ERR_TIMEOUT in the device status word; te_get_device_status reads and clears it;
and the context keeps working afterwards (a bit-exact E4M3 cast through the library).
"""

import time

import numpy as np
import pytest
import torch

import fp8_transformer_gb300 as te
from oracle import numerics as nx
from parity import codes, np64
from workloads import random_tensor

pytestmark = pytest.mark.gpu


def test_timed_out_wait_is_reported_and_the_context_survives():
    torch.cuda.synchronize()
    assert te.get_device_status() == te.binding.TE_OK  # nothing pending (and cleared)
    t0 = time.perf_counter()
    te.selftest_wait_timeout(20000)
    assert te.get_device_status() == te.binding.TE_ERR_TIMEOUT
    assert time.perf_counter() - t0 >= 0.02  # the wait ran for its whole limit
    assert te.get_device_status() == te.binding.TE_OK  # read and cleared
    x = random_tensor((256, 512), device="cuda", seed=3)
    q = te.Quantizer(64.0)
    out = torch.empty(256, 512, dtype=torch.uint8, device="cuda")
    te.te_quantize(x, q, out)
    torch.cuda.synchronize()
    want = nx.quantize(nx.to_f32(np64(x)), np.float32(64.0))
    assert np.array_equal(codes(out), want)
    assert te.get_device_status() == te.binding.TE_OK
