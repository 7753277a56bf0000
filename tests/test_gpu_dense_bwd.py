"""Backward of LayerNorm -> Dense (te_layernorm_dense_bwd) against the oracle.

The GPU runs its own forward (te_layernorm_dense_fwd, keeping the normalized output, mu and
rsigma) and then the backward.  Those saved tensors, dy, x, gamma and the kernel are the
backward call's inputs; the oracle's steps start from them (``steps.check_dense_bwd``) and hold
each output to the pages' rules: dbias (column sums of the identical dy) to 1e-4; dkernel and
the dln inside the call as GEMM outputs whose bf16 rounding may differ only where the fp32
accumulation window straddles a midpoint; dx, dgamma, dbeta to the reduction / bf16 rules plus
the window that dln's rounding can explain.  In FP8 mode dy and the kernel are cast from
identical inputs (their scales checked exactly), so their codes are the oracle's.
"""

import numpy as np
import pytest
import torch

import fp8_transformer_gb300 as te
from oracle import numerics as nx
from parity import assert_in_window, codes, decode, np64, quantize_fast
from steps import check_dense_bwd, check_norm_dx, check_norm_params, gemm_ref
from workloads import make_inputs, random_tensor

pytestmark = pytest.mark.gpu
DEV = "cuda"
SCALES = dict(x=32.0, kernel=2048.0, grad=16.0)


def quantizers(mode):
    if mode is None:
        return None
    if mode == "delayed":
        return te.QuantizerSet(x=te.Quantizer(SCALES["x"]), kernel1=te.Quantizer(SCALES["kernel"]),
                               grad=te.Quantizer(SCALES["grad"]))
    return te.QuantizerSet(x=te.Quantizer(mode="current"), kernel1=te.Quantizer(mode="current"),
                           grad=te.Quantizer(mode="current"))


def run_gpu(inp, dy, mode):
    M, H, N = inp["M"], inp["H"], inp["N"]
    dt = torch.bfloat16
    qs = quantizers(mode)
    out = torch.empty(M, N, dtype=dt, device=DEV)
    ln = torch.empty(M, H, dtype=torch.uint8 if mode else dt, device=DEV)
    mu = torch.empty(M, dtype=torch.float32, device=DEV)
    rs = torch.empty(M, dtype=torch.float32, device=DEV)
    kw = dict(norm_type=inp["norm"], zero_centered_gamma=inp["zero_centered_gamma"])
    te.te_layernorm_dense_fwd(inp["x"], inp["kernel"], inp["gamma"], inp["beta"], inp.get("bias"),
                              out, epsilon=inp["eps"], saved_ln_out=ln, mu=mu, rsigma=rs,
                              quantizer_set=qs, **kw)
    g = dict(dx=torch.empty(M, H, dtype=dt, device=DEV),
             dgamma=torch.empty(H, dtype=torch.float32, device=DEV),
             dbeta=torch.empty(H, dtype=torch.float32, device=DEV),
             dkernel=torch.empty(H, N, dtype=dt, device=DEV),
             dbias=torch.empty(N, dtype=torch.float32, device=DEV))
    te.te_layernorm_dense_bwd(dy, inp["x"], inp["gamma"], inp["kernel"], ln, mu, rs, g["dx"],
                              g["dgamma"], g["dkernel"], dbeta=g["dbeta"], dbias=g["dbias"],
                              quantizer_set=qs, **kw)
    torch.cuda.synchronize()
    g.update(qs=qs, ln=ln, mu=mu, rs=rs)
    if inp["norm"] != "layernorm":  # no shift: the gradient of the unused beta is zero
        assert int(g["dbeta"].count_nonzero().item()) == 0
        g["dbeta"] = None
    return g, qs


def dense_inputs(M, H, N, norm="layernorm", zc=False, seed=0):
    inp = make_inputs("qkv_ln_dense", device=DEV, M=M, H=H, N=N, seed=seed)
    inp["norm"] = norm
    inp["zero_centered_gamma"] = zc
    if zc:
        inp["gamma"] = random_tensor((H,), std=0.05, device=DEV, seed=seed + 7)
    return inp


CASES = [dict(M=300, H=512, N=784), dict(M=256, H=272, N=528)]


@pytest.mark.parametrize("shape", CASES)
@pytest.mark.parametrize("mode", [None, "delayed", "current"])
@pytest.mark.parametrize("norm,zc", [("layernorm", False), ("rmsnorm", True)])
def test_dense_backward_small(shape, mode, norm, zc):
    inp = dense_inputs(**shape, norm=norm, zc=zc)
    M, H, N = inp["M"], inp["H"], inp["N"]
    dy = random_tensor((M, N), device=DEV, seed=5)
    g, qs = run_gpu(inp, dy, mode)
    if mode == "current":
        # dy and the kernel are identical inputs: their amaxes, hence their scales, are exact
        for q, t in ((qs.grad, np64(dy)), (qs.kernel1, np64(inp["kernel"]))):
            assert np.float32(q.amax.item()) == nx.amax_of(t)
            assert np.float32(q.scale.item()) == nx.compute_scale(nx.amax_of(t))[0]
        assert np.float32(qs.x.scale.item()) == nx.compute_scale(np.float32(qs.x.amax.item()))[0]
    elif mode == "delayed":
        assert qs.grad.scale.item() == SCALES["grad"]
    check_dense_bwd(np64(dy), np64(inp["x"]), np64(inp["gamma"]), np64(inp["kernel"]), g,
                    mode is not None, norm, zc)


def test_dense_backward_no_tokens():
    """M = 0: every gradient comes back zero (the buffers start as NaN)."""
    H, N = 64, 96
    x = torch.empty(0, H, dtype=torch.bfloat16, device=DEV)
    dy = torch.empty(0, N, dtype=torch.bfloat16, device=DEV)
    gamma = torch.ones(H, dtype=torch.bfloat16, device=DEV)
    kernel = torch.ones(H, N, dtype=torch.bfloat16, device=DEV)
    empty = torch.empty(0, dtype=torch.float32, device=DEV)
    dgamma = torch.full((H,), float("nan"), device=DEV)
    dbeta = torch.full((H,), float("nan"), device=DEV)
    dbias = torch.full((N,), float("nan"), device=DEV)
    dk = torch.full((H, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    te.te_layernorm_dense_bwd(dy, x, gamma, kernel, x, empty, empty, x, dgamma, dk, dbeta=dbeta,
                              dbias=dbias)
    torch.cuda.synchronize()
    for t in (dgamma, dbeta, dbias, dk):
        assert torch.count_nonzero(t).item() == 0


@pytest.mark.parametrize("mode", [None, "delayed"])
def test_dense_backward_full_size_sampled(mode):
    """The full QKV shape (16384 tokens, 8192 -> 24576), bf16 and FP8 (delayed scaling), in the
    launch configuration the benchmark times.  The oracle's steps run from the backward's
    inputs on a sample: rows of dx (row-local), columns of dkernel and dbias (one dy column
    each) and columns of dgamma / dbeta (dln over every token)."""
    inp = make_inputs("qkv_ln_dense", device=DEV)
    M, H, N = inp["M"], inp["H"], inp["N"]
    dy = random_tensor((M, N), device=DEV, seed=9)
    g, qs = run_gpu(inp, dy, mode)
    for k in ("dx", "dgamma", "dbeta", "dkernel", "dbias"):
        assert torch.isfinite(g[k].float()).all(), k
    fp8 = mode is not None
    rng = np.random.default_rng(13)
    cols = np.sort(rng.choice(N, 6, replace=False))
    cols[-1] = N - 1
    rows = np.array([0, 1, 100, 5000, 12345, M - 1])          # rows 0 and 100 are x8 rows
    hcols = np.sort(rng.choice(H, 5, replace=False))
    dy_c = np64(dy[:, torch.as_tensor(cols, device=DEV)])
    assert_in_window(np64(g["dbias"])[cols], dy_c.sum(axis=0), 0.0, "dbias columns")
    kern = np64(inp["kernel"])
    x64 = np64(inp["x"])
    gamma = np64(inp["gamma"])
    mu, rs = np64(g["mu"]), np64(g["rs"])
    if fp8:
        s_g = np.float32(qs.grad.scale.item())
        s_k = np.float32(qs.kernel1.scale.item())
        q = lambda v, s: decode(quantize_fast(v, s))
        ln = decode(codes(g["ln"]))
        a_dk = float(np.float32(qs.x.scale_inv.item()) * np.float32(qs.grad.scale_inv.item()))
        a_dln = float(np.float32(qs.grad.scale_inv.item()) * np.float32(qs.kernel1.scale_inv.item()))
    else:
        q = lambda v, s: v
        s_g = s_k = None
        ln, a_dk, a_dln = np64(g["ln"]), 1.0, 1.0
    dk, w_dk = gemm_ref(ln.T, q(dy_c, s_g), a_dk)                       # [H, 6]
    assert_in_window(np64(g["dkernel"])[:, cols], dk, w_dk, "dkernel columns", stored="bf16")
    kq = q(kern, s_k)
    dy_r = np64(dy[torch.as_tensor(rows, device=DEV)])
    dln_r, w_r = gemm_ref(q(dy_r, s_g), kq.T, a_dln)
    check_norm_dx(np64(g["dx"])[rows], dln_r, w_r, x64[rows], mu[rows], rs[rows], gamma,
                  "layernorm", False, what="dx rows")
    # dln[:, hcols] over every token, in row chunks
    kc = kq[hcols].T
    parts, wparts = [], []
    for r0 in range(0, M, 2048):
        d = q(np64(dy[r0:r0 + 2048]), s_g)
        v, w = gemm_ref(d, kc, a_dln)
        parts.append(v)
        wparts.append(w)
    check_norm_params(np64(g["dgamma"])[hcols], np64(g["dbeta"])[hcols], np.concatenate(parts),
                      np.concatenate(wparts), x64[:, hcols], mu, rs, "layernorm",
                      what="norm columns")
