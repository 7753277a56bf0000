"""The data-parallel helpers on one GPU: te_update_scales against the recipe, and the
bucketed backward (one-rank NCCL group) against te_layernorm_mlp_bwd itself.

The two-rank exchanges are covered on the CPU by tests/test_dist_gloo.py.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist

import fp8_transformer_gb300 as te
from fp8_transformer_gb300 import dp
from oracle import numerics as nx
from workloads import make_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_update_scales_follows_the_recipe():
    """scale = fp32(448 / amax), with scale 1 for amax 0 / inf / NaN and FLT_MAX when the
    quotient overflows; scale_inv = fp32(1 / scale); disabled quantizers are skipped."""
    amaxes = [3.0, 0.0, float("inf"), float("nan"), 1e-40, 448.0, 0.1, 7e5]
    qs = []
    for a in amaxes:
        q = te.Quantizer(5.0)
        q.amax.fill_(a)
        qs.append(q)
    te.te_update_scales(qs)
    torch.cuda.synchronize()
    for a, q in zip(amaxes, qs):
        s, si = nx.compute_scale(np.float32(a))
        assert np.float32(q.scale.item()) == s, a
        assert np.float32(q.scale_inv.item()) == si, a


def test_update_scales_rejects_bad_arguments():
    with pytest.raises(te.TEError) as e:
        te.te_update_scales([te.Quantizer(1.0) for _ in range(17)])
    assert e.value.status == te.binding.TE_ERR_INVALID_ARG


def _one_rank_group():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("nccl", rank=0, world_size=1)


@pytest.mark.parametrize("fp8", [False, True])
def test_bucketed_backward_one_rank(fp8):
    """With one rank the sum over ranks is the identity: the bucketed backward must give the
    plain call's gradients bit for bit, and the bank's amax exchange and scale update the
    recipe's scales."""
    inp = make_inputs("gpt_ln_mlp_bwd", device=DEV, M=300, H=512, F=784)
    M, H, F = inp["M"], inp["H"], inp["F"]
    bank = dp.QuantizerBank(dict(x=32.0, kernel1=2048.0, act=16.0, kernel2=2048.0, grad=64.0),
                            device=DEV)
    qs = bank.quantizer_set() if fp8 else None
    out = torch.empty(M, H, dtype=torch.bfloat16, device=DEV)
    h = torch.empty(M, F, dtype=torch.bfloat16, device=DEV)
    ln = torch.empty(M, H, dtype=torch.uint8 if fp8 else torch.bfloat16, device=DEV)
    mu = torch.empty(M, dtype=torch.float32, device=DEV)
    rs = torch.empty(M, dtype=torch.float32, device=DEV)
    kw = dict(norm_type="layernorm", activation_type="gelu", quantizer_set=qs)
    te.te_layernorm_mlp_fwd(inp["x"], inp["gamma"], inp["beta"], inp["w1"], inp["w2"], inp["b1"],
                            inp["b2"], out, epsilon=inp["eps"], saved_h=h, saved_ln_out=ln, mu=mu,
                            rsigma=rs, **kw)
    ref = dict(dx=torch.empty(M, H, dtype=torch.bfloat16, device=DEV),
               dg=torch.empty(H, device=DEV), db=torch.empty(H, device=DEV),
               dw1=torch.empty(H, F, dtype=torch.bfloat16, device=DEV),
               dw2=torch.empty(F, H, dtype=torch.bfloat16, device=DEV),
               db1=torch.empty(F, device=DEV), db2=torch.empty(H, device=DEV))
    te.te_layernorm_mlp_bwd(inp["dy"], inp["x"], inp["gamma"], inp["w1"], inp["w2"], h, ln, mu,
                            rs, ref["dx"], ref["dg"], ref["dw1"], ref["dw2"], dbeta=ref["db"],
                            dbias1=ref["db1"], dbias2=ref["db2"], **kw)
    _one_rank_group()
    try:
        b = dp.GradBuckets(H, F, False, device=DEV)
        dx = torch.empty(M, H, dtype=torch.bfloat16, device=DEV)
        dp.layernorm_mlp_bwd_dp(inp["dy"], inp["x"], inp["gamma"], inp["w1"], inp["w2"], h, ln,
                                mu, rs, dx, b, **kw)
        amax_before = bank.amax.clone()
        bank.allreduce_amax()
        bank.update_scales()
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    assert torch.equal(dx, ref["dx"])
    for got, want in ((b.dkernel1, ref["dw1"]), (b.dkernel2, ref["dw2"]), (b.dgamma, ref["dg"]),
                      (b.dbeta, ref["db"]), (b.dbias1, ref["db1"]), (b.dbias2, ref["db2"])):
        assert torch.equal(got, want)
    assert torch.equal(bank.amax, amax_before)
    if fp8:
        for i, n in enumerate(dp.NAMES):
            s, si = nx.compute_scale(np.float32(bank.amax[i].item()))
            assert np.float32(bank.scale[i].item()) == s, n
            assert np.float32(bank.scale_inv[i].item()) == si, n
