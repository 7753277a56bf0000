"""Backward of LayerNorm -> Dense (te_layernorm_dense_bwd) against the oracle.

The GPU runs its own forward (te_layernorm_dense_fwd, keeping the normalized output, mu and
rsigma) and then the backward; the oracle runs its own forward and backward from the same x,
kernel and upstream gradient.  Rules:

* dbias = column sums of dy (identical inputs on both sides): the 1e-4 reduction rule;
* dkernel (a contraction over tokens): the GEMM rule, with the one-flip term when the
  normalized output is a self-computed E4M3 operand;
* dx, dgamma, dbeta, which carry the dln GEMM's error: 4e-2 / 2e-2 of their magnitude.
"""

import numpy as np
import pytest
import torch

import fp8_transformer_gb300 as te
from oracle import block as ob
from oracle import numerics as nx
from parity import assert_gemm_close, assert_reduction_close, np64, rms
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
    return g, qs


def close(got, ref, what, rel=2e-2):
    got, ref = np64(got), np.asarray(ref, np.float64)
    tol = rel * np.maximum(np.abs(ref), rms(ref)) + 2.0 ** -8 * np.abs(ref)
    bad = np.abs(got - ref) > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outside; worst "
                           f"{float((np.abs(got - ref) / tol).max()):.2f}x")


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
    f = lambda k: None if inp.get(k) is None else np64(inp[k])
    fp8 = None
    if mode == "delayed":
        fp8 = {k: np.float32(v) for k, v in SCALES.items()}
    elif mode == "current":
        # the normalized output's scale comes from the GPU's own amax (of its fp32 norm output);
        # the oracle quantizes its normalized output with that scale, so that the two sets of
        # codes differ only by flips at rounding boundaries
        amax = np.float32(qs.x.amax.item())
        assert np.float32(qs.x.scale.item()) == nx.compute_scale(amax)[0]
        fp8 = dict(x=np.float32(qs.x.scale.item()), kernel=None, grad=None)
    ref = ob.layernorm_dense_bwd(np64(dy), f("x"), f("gamma"), f("beta"), f("kernel"), f("bias"),
                                 norm, zc, inp["eps"], "bf16", fp8=fp8)
    if mode == "current":
        assert abs(float(amax) - float(ref["fwd"]["ln"].amax)) <= 1e-5 * float(amax)
        # dy and the kernel are identical inputs: their amax, hence their scales, are identical
        assert np.float32(qs.grad.scale.item()) == ref["dy"].scale
        assert np.float32(qs.kernel1.scale.item()) == ref["fwd"]["kernel"].scale
    assert_reduction_close(g["dbias"], ref["dbias"], what="dbias")
    ln = ref["fwd"]["ln"].value * ref["fwd"]["ln"].inv()
    gy = ref["dy"].value * ref["dy"].inv()
    assert_gemm_close(g["dkernel"], ref["dkernel"].value, M, rms(ln), rms(gy), what="dkernel",
                      fp8_operands=(ln.T, gy) if mode else None)
    close(g["dx"], ref["dx"].value, "dx", rel=4e-2)
    close(g["dgamma"], ref["dgamma"], "dgamma")
    if norm == "layernorm":
        close(g["dbeta"], ref["dbeta"], "dbeta")


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


def test_dense_backward_full_size_sampled():
    """The full QKV shape (16384 tokens, 8192 -> 24576), bf16.  The oracle recomputes, from
    its own primitives and in float64, rows of dx (row-local), columns of dkernel and dbias
    (one dy column each)."""
    inp = make_inputs("qkv_ln_dense", device=DEV)
    M, H, N = inp["M"], inp["H"], inp["N"]
    dy = random_tensor((M, N), device=DEV, seed=9)
    g, _ = run_gpu(inp, dy, None)
    for k, v in g.items():
        assert torch.isfinite(v.float()).all(), k
    bf = lambda v: nx.bf16_round(nx.to_f32(v))
    rng = np.random.default_rng(13)
    cols = np.sort(rng.choice(N, 6, replace=False))
    dy_c = np64(dy[:, torch.as_tensor(cols, device=DEV)])
    assert_reduction_close(np64(g["dbias"])[cols], dy_c.sum(axis=0), what="dbias sampled")
    x64 = np64(inp["x"])
    gamma, beta = np64(inp["gamma"]), np64(inp["beta"])
    y, mu, rs = ob.norm_fwd(x64, gamma, beta, "layernorm", False, inp["eps"])
    ln = bf(y)
    dk_ref = bf(ln.T @ dy_c)                                   # [H, 6]
    assert_gemm_close(np64(g["dkernel"])[:, cols], dk_ref, M, rms(ln), rms(dy_c),
                      what="dkernel columns", stored="bf16")
    rows = np.array([0, 1, 100, 5000, 12345, M - 1])          # rows 0 and 100 are x8 rows
    kern = np64(inp["kernel"])
    dln_r = bf(np64(dy[torch.as_tensor(rows, device=DEV)]) @ kern.T)
    dx_r, _, _ = ob.norm_bwd(dln_r, x64[rows], mu[rows], rs[rows], gamma, "layernorm", False)
    close(np64(g["dx"])[rows], bf(dx_r), "dx rows", rel=4e-2)
