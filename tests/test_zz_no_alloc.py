"""te_dact_dbias_quantize_noalloc against te_dact_dbias_quantize, through the C ABI.

The no-allocation variant serves callers that cannot give the library a workspace (runtimes
that plan all device memory up front, latency-critical code that cannot afford cudaMalloc's
device-wide synchronization).  It must produce what the workspace version produces, also on a
second call in a row (its fixed scratch keeps the previous call's contents), and refuse sizes
beyond its fixed capacity.  This file is collected last so that a failure here cannot hide
another test's result.
"""

import numpy as np
import pytest
import torch

import fp8_transformer_gb300 as te
from oracle import block as ob
from oracle import numerics as nx
from parity import assert_e4m3_codes, assert_reduction_close, np64
from workloads import random_tensor

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(M, N_in, act, seed):
    n_out = N_in // 2 if act == "swiglu" else N_in
    dy = random_tensor((M, n_out), device=DEV, seed=seed)
    h = random_tensor((M, N_in), std=2.0, device=DEV, seed=seed + 1)
    return dy, h


@pytest.mark.parametrize("act,M,N_in,fp8", [("gelu", 1000, 4096, False),
                                            ("swiglu", 777, 2048, True),
                                            ("gelu", 2048, 1024, True)])
def test_noalloc_matches_workspace_version_twice(act, M, N_in, fp8):
    for call, seed in enumerate((11, 23)):  # two calls in a row, different data
        dy, h = _inputs(M, N_in, act, seed)
        out_dt = torch.uint8 if fp8 else torch.bfloat16
        dx_ref = torch.empty(M, N_in, dtype=out_dt, device=DEV)
        db_ref = torch.empty(N_in, dtype=torch.float32, device=DEV)
        dx_new = torch.full((M, N_in), 7, dtype=out_dt, device=DEV)
        db_new = torch.full((N_in,), 123.0, dtype=torch.float32, device=DEV)
        q_ref = te.Quantizer(16.0) if fp8 else None
        q_new = te.Quantizer(16.0) if fp8 else None
        te.te_dact_dbias_quantize(dy, h, act, dx_ref, dbias=db_ref, q=q_ref)
        te.te_dact_dbias_quantize_noalloc(dy, h, act, dx_new, dbias=db_new, q=q_new)
        torch.cuda.synchronize()
        # the same kernels in the same summation order: bit for bit, whatever the first call
        # left in the fixed scratch
        if fp8:
            assert_e4m3_codes(dx_new, np64(dx_ref), what=f"dx call {call}")
            assert q_new.amax.item() == q_ref.amax.item()
            assert q_new.scale_inv.item() == q_ref.scale_inv.item()
        else:
            assert torch.equal(dx_new, dx_ref), f"dx call {call}"
        assert torch.equal(db_new, db_ref), f"dbias call {call}"
        # and both within the reduction rule of the oracle's column sums
        ref = ob.act_bwd(np64(dy), np64(h), act)
        assert_reduction_close(db_new, ob.colsum(nx.to_f32(ref)), what=f"dbias call {call}")


def test_noalloc_current_scaling_matches():
    dy, h = _inputs(512, 1024, "gelu", 5)
    res = []
    for fn in (te.te_dact_dbias_quantize, te.te_dact_dbias_quantize_noalloc):
        dx = torch.empty(512, 1024, dtype=torch.uint8, device=DEV)
        db = torch.empty(1024, dtype=torch.float32, device=DEV)
        q = te.Quantizer(1.0, mode="current")
        fn(dy, h, "gelu", dx, dbias=db, q=q)
        torch.cuda.synchronize()
        res.append((np64(dx), np64(db), q.scale.item(), q.amax.item()))
    assert np.array_equal(res[0][0], res[1][0])
    assert np.array_equal(res[0][1], res[1][1])
    assert res[0][2] == res[1][2] and res[0][3] == res[1][3]


def test_noalloc_rejects_sizes_beyond_capacity():
    cap = te.dact_dbias_noalloc_capacity()
    N_in = 16384
    rows_ok = (cap // N_in) * 128  # partial rows of 128 tokens fill the capacity exactly
    dy = torch.empty(rows_ok + 128, N_in, dtype=torch.bfloat16, device=DEV)
    dx = torch.empty_like(dy)
    db = torch.empty(N_in, dtype=torch.float32, device=DEV)
    with pytest.raises(te.TEError) as e:
        te.te_dact_dbias_quantize_noalloc(dy, None, "identity", dx, dbias=db)
    assert e.value.status == te.binding.TE_ERR_TOO_LARGE
    # without dbias nothing is reduced and no scratch is needed
    small = dy[:256]
    te.te_dact_dbias_quantize_noalloc(small, None, "identity", dx[:256])
    torch.cuda.synchronize()
    assert torch.equal(dx[:256], small)
