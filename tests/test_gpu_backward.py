"""Backward of the LayerNorm-MLP block (te_layernorm_mlp_bwd) against the oracle.

The GPU runs its own forward (te_layernorm_mlp_fwd, keeping h, the normalized output, mu and
rsigma) and then the backward; the oracle runs its own forward and backward from the same x,
weights and upstream gradient.  Every gradient is compared:

* weight gradients (contraction over tokens) and the pre-norm gradient by the GEMM rule
  (2e-2 of the expected magnitude, plus one bf16 ulp of the stored value);
* bias and gain gradients, whose inputs carry that GEMM error, to 2e-2 of their magnitude;
* dbias2 = column sums of dy (identical inputs on both sides) to the 1e-4 reduction rule.
"""

import numpy as np
import pytest
import torch

import fp8_transformer_gb300 as te
from oracle import block as ob
from oracle import numerics as nx
from parity import assert_gemm_close, assert_reduction_close, np64, rms
from workloads import make_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
SCALES = dict(x=32.0, w1=2048.0, act=16.0, w2=2048.0, grad=64.0)


def run_gpu(inp, fp8, mode="delayed", keep=None):
    """GPU forward + backward; `keep` (a dict) receives the quantizer set."""
    M, H, F = inp["M"], inp["H"], inp["F"]
    gated = ob.GATED[inp["act"]]
    F1 = 2 * F if gated else F
    dt = torch.bfloat16
    qs = None
    if fp8 and mode == "delayed":
        qs = te.QuantizerSet(x=te.Quantizer(SCALES["x"]), kernel1=te.Quantizer(SCALES["w1"]),
                             act=te.Quantizer(SCALES["act"]), kernel2=te.Quantizer(SCALES["w2"]),
                             grad=te.Quantizer(SCALES["grad"]))
    elif fp8:
        qs = te.QuantizerSet(**{k: te.Quantizer(mode="current")
                                for k in ("x", "kernel1", "act", "kernel2", "grad")})
    if keep is not None:
        keep["qs"] = qs
    out = torch.empty(M, H, dtype=dt, device=DEV)
    h = torch.empty(M, F1, dtype=dt, device=DEV)
    ln = torch.empty(M, H, dtype=torch.uint8 if fp8 else dt, device=DEV)
    mu = torch.empty(M, dtype=torch.float32, device=DEV)
    rs = torch.empty(M, dtype=torch.float32, device=DEV)
    kw = dict(norm_type=inp["norm"], zero_centered_gamma=inp["zero_centered_gamma"],
              activation_type=inp["act"], quantizer_set=qs)
    te.te_layernorm_mlp_fwd(inp["x"], inp["gamma"], inp["beta"], inp["w1"], inp["w2"],
                            inp.get("b1"), inp.get("b2"), out, epsilon=inp["eps"], saved_h=h,
                            saved_ln_out=ln, mu=mu, rsigma=rs, **kw)
    g = dict(dx=torch.empty(M, H, dtype=dt, device=DEV),
             dgamma=torch.empty(H, dtype=torch.float32, device=DEV),
             dbeta=torch.empty(H, dtype=torch.float32, device=DEV),
             dw1=torch.empty(H, F1, dtype=dt, device=DEV),
             dw2=torch.empty(F, H, dtype=dt, device=DEV),
             db1=torch.empty(F1, dtype=torch.float32, device=DEV),
             db2=torch.empty(H, dtype=torch.float32, device=DEV))
    te.te_layernorm_mlp_bwd(inp["dy"], inp["x"], inp["gamma"], inp["w1"], inp["w2"], h, ln, mu, rs,
                            g["dx"], g["dgamma"], g["dw1"], g["dw2"], dbeta=g["dbeta"],
                            dbias1=g["db1"], dbias2=g["db2"], **kw)
    torch.cuda.synchronize()
    return g


def run_oracle(inp, fp8, scales=None):
    f = lambda k: None if inp.get(k) is None else np64(inp[k])
    sc = scales if scales is not None else {k: np.float32(v) for k, v in SCALES.items()}
    return ob.layernorm_mlp_bwd(f("dy"), f("x"), f("gamma"), f("beta"), f("w1"), f("w2"),
                                f("b1"), f("b2"), inp["norm"], inp["zero_centered_gamma"],
                                inp["eps"], inp["act"], "bf16", fp8=sc if fp8 else None)


def close(got, ref, what, rel=2e-2):
    got, ref = np64(got), np.asarray(ref, np.float64)
    tol = rel * np.maximum(np.abs(ref), rms(ref)) + 2.0 ** -8 * np.abs(ref)
    bad = np.abs(got - ref) > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outside; worst "
                           f"{float((np.abs(got - ref) / tol).max()):.2f}x")


def check(inp, g, ref):
    M = inp["M"]
    fwd = ref["fwd"]
    assert_reduction_close(g["db2"], ref["db2"], what="dbias2")
    a = ref["a_re"].value
    assert_gemm_close(g["dw2"], ref["dW2"].value, M, rms(a), rms(np64(inp["dy"])), what="dW2")
    ln = fwd["ln"].value * fwd["ln"].inv()
    dh = ref["dh"].value * ref["dh"].inv()
    fp8 = ref["dh"].dtype == "e4m3"
    assert_gemm_close(g["dw1"], ref["dW1"].value, M, rms(ln), rms(dh), what="dW1",
                      fp8_operands=(ln.T, dh) if fp8 else None)
    close(g["db1"], ref["db1"], "dbias1")
    close(g["dx"], ref["dx"].value, "dx", rel=4e-2)
    close(g["dgamma"], ref["dgamma"], "dgamma")
    if inp["norm"] == "layernorm":
        close(g["dbeta"], ref["dbeta"], "dbeta")


CASES = [("gpt_ln_mlp_bwd", dict(M=300, H=512, F=784)),
         ("llama_rms_mlp", dict(M=256, H=512, F=528))]


def _inputs(name, shape):
    inp = make_inputs(name, device=DEV, **shape)
    if "dy" not in inp:  # the Llama case draws its upstream gradient after its own tensors
        inp["dy"] = make_inputs("gpt_ln_mlp_bwd", device=DEV, M=inp["M"], H=inp["H"], F=16,
                                seed=1)["dy"]
    return inp


@pytest.mark.parametrize("name,shape", CASES)
@pytest.mark.parametrize("fp8", [False, True])
def test_mlp_backward_small(name, shape, fp8):
    inp = _inputs(name, shape)
    g = run_gpu(inp, fp8)
    ref = run_oracle(inp, fp8)
    check(inp, g, ref)


@pytest.mark.parametrize("name,shape", CASES)
def test_mlp_backward_fp8_current_scaling(name, shape):
    """Every quantizer in current scaling: the forward's casts and the backward's dH cast each
    take a separate amax pass (the dbias reduction runs in dH's amax pass).  The normalized
    output, the activation output and dH are computed by each side itself, so the oracle
    quantizes them with the GPU's scales, after checking that each scale is the recipe's
    function of the GPU's amax and that the amaxes agree; the weights' scales come from
    identical inputs and must be identical."""
    inp = _inputs(name, shape)
    keep = {}
    g = run_gpu(inp, True, mode="current", keep=keep)
    qs = keep["qs"]
    gpu_scale = {}
    for name_q, q in (("x", qs.x), ("act", qs.act), ("grad", qs.grad)):
        amax = np.float32(q.amax.item())
        assert np.float32(q.scale.item()) == nx.compute_scale(amax)[0], name_q
        gpu_scale[name_q] = np.float32(q.scale.item())
    ref = run_oracle(inp, True, scales=dict(x=gpu_scale["x"], w1=None, act=gpu_scale["act"],
                                            w2=None, grad=gpu_scale["grad"]))
    assert np.float32(qs.kernel1.scale.item()) == ref["fwd"]["w1"].scale
    assert np.float32(qs.kernel2.scale.item()) == ref["fwd"]["w2"].scale
    assert abs(qs.x.amax.item() - float(ref["fwd"]["ln"].amax)) <= 1e-5 * float(ref["fwd"]["ln"].amax)
    assert abs(qs.act.amax.item() - float(ref["fwd"]["a"].amax)) <= 2e-2 * float(ref["fwd"]["a"].amax)
    assert abs(qs.grad.amax.item() - float(ref["dh"].amax)) <= 2e-2 * float(ref["dh"].amax)
    check(inp, g, ref)


@pytest.mark.parametrize("act", ["geglu", "reglu"])
@pytest.mark.parametrize("fp8", [False, True])
def test_mlp_backward_other_gated(act, fp8):
    """("gelu", "linear") and ("relu", "linear"): the recomputed activation, the gated
    dact + dbias (+ E4M3) step and the rest of the backward."""
    inp = _inputs("llama_rms_mlp", dict(M=256, H=512, F=528))
    inp["act"] = act
    g = run_gpu(inp, fp8)
    ref = run_oracle(inp, fp8)
    check(inp, g, ref)


def test_mlp_backward_full_size_sampled():
    """The full GPT backward (16384 tokens, 4096 -> 16384 -> 4096, gelu), bf16.  The oracle
    recomputes, from its own primitives and in float64, what a sample of outputs depends on:
    rows of dx (row-local), rows of dW2 (one GEMM1 column each), columns of dW1 and dbias1 (one
    dA column each), and all of dbias2."""
    inp = make_inputs("gpt_ln_mlp_bwd", device=DEV)
    g = run_gpu(inp, fp8=False)
    for k, v in g.items():
        assert torch.isfinite(v.float()).all(), k
    M, H, F = inp["M"], inp["H"], inp["F"]
    f64 = lambda k: np64(inp[k])
    x, gamma, beta, w1, w2, b1, b2, dy = (f64(k) for k in ("x", "gamma", "beta", "w1", "w2", "b1",
                                                           "b2", "dy"))
    bf = lambda v: nx.bf16_round(nx.to_f32(v))
    assert_reduction_close(g["db2"], ob.colsum(dy), what="dbias2")
    # normalized operand of every token (needed by the column samples)
    y, mu, rs = ob.norm_fwd(x, gamma, beta, "layernorm", False, inp["eps"])
    ln = bf(y)
    rng = np.random.default_rng(11)
    # rows of dx: everything row-local
    rows = np.sort(rng.choice(M, 12, replace=False))
    h_r = bf(ob.gemm(ln[rows], w1, b1))
    da_r = bf(ob.gemm(dy[rows], w2.T))
    dh_r = bf(ob.act_bwd(da_r, h_r, "gelu"))
    dln_r = bf(ob.gemm(dh_r, w1.T))
    dx_r, _, _ = ob.norm_bwd(dln_r, x[rows], mu[rows], rs[rows], gamma, "layernorm", False)
    close(np64(g["dx"])[rows], bf(dx_r), "dx rows", rel=4e-2)
    # columns f of the hidden layer: dW2[f, :], dW1[:, f], dbias1[f]
    feats = np.sort(rng.choice(F, 6, replace=False))
    h_c = bf(ln @ w1[:, feats] + b1[feats])            # [M, 6]
    a_c = bf(ob.act_fwd(h_c, "gelu"))
    dw2_ref = bf(a_c.T @ dy)                           # [6, H]
    assert_gemm_close(np64(g["dw2"])[feats], dw2_ref, M, rms(a_c), rms(dy), what="dW2 rows",
                      stored="bf16")
    da_c = bf(dy @ w2[feats].T)                        # [M, 6]
    dh_c = nx.to_f32(ob.act_bwd(da_c, h_c, "gelu"))
    close(np64(g["db1"])[feats], dh_c.sum(axis=0), "dbias1 sampled")
    dw1_ref = bf(ln.T @ bf(dh_c))                      # [H, 6]
    assert_gemm_close(np64(g["dw1"])[:, feats], dw1_ref, M, rms(ln), rms(dh_c),
                      what="dW1 columns", stored="bf16")
