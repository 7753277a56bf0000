"""Backward of the LayerNorm-MLP block (te_layernorm_mlp_bwd) against the oracle.

The GPU runs its own forward (te_layernorm_mlp_fwd, keeping h, the normalized output, mu and
rsigma) and then the backward, with dH kept through ``saved_dh``.  The saved tensors are the
backward call's inputs, so the oracle's steps start from them and each output is held to the
pages' rules step by step (``steps``): fp32 reductions to 1e-4, E4M3 codes and amax exact up to
the rounding of the step's own fp32 arithmetic, bf16 values up to the rounding of an fp32
intermediate, each plus only the window that the rounding of the chain's fp32 intermediates
can explain.
"""

import numpy as np
import pytest
import torch

import fp8_transformer_gb300 as te
from oracle import block as ob
from oracle import numerics as nx
from parity import (ACC_REL, Guarded, assert_in_window, bf16_jump, codes, decode, np64,
                    quantize_fast)
from steps import (ACT_REL, SCALE_REL, check_dact, check_mlp_bwd, check_norm_dx,
                   check_norm_params, gemm_ref)
from workloads import make_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
SCALES = dict(x=32.0, w1=2048.0, act=16.0, w2=2048.0, grad=64.0)


def run_gpu(inp, fp8, mode="delayed"):
    """GPU forward + backward; returns the saved tensors, the gradients, dH and the quantizers."""
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
    out = torch.empty(M, H, dtype=dt, device=DEV)
    g = dict(qs=qs, h=torch.empty(M, F1, dtype=dt, device=DEV),
             ln=torch.empty(M, H, dtype=torch.uint8 if fp8 else dt, device=DEV),
             mu=torch.empty(M, dtype=torch.float32, device=DEV),
             rs=torch.empty(M, dtype=torch.float32, device=DEV))
    kw = dict(norm_type=inp["norm"], zero_centered_gamma=inp["zero_centered_gamma"],
              activation_type=inp["act"], quantizer_set=qs)
    te.te_layernorm_mlp_fwd(inp["x"], inp["gamma"], inp["beta"], inp["w1"], inp["w2"],
                            inp.get("b1"), inp.get("b2"), out, epsilon=inp["eps"], saved_h=g["h"],
                            saved_ln_out=g["ln"], mu=g["mu"], rsigma=g["rs"], **kw)
    guards = dict(dx=Guarded((M, H), dt), dgamma=Guarded((H,), torch.float32),
                  dbeta=Guarded((H,), torch.float32), dw1=Guarded((H, F1), dt),
                  dw2=Guarded((F, H), dt), db1=Guarded((F1,), torch.float32),
                  db2=Guarded((H,), torch.float32),
                  dh=Guarded((M, F1), torch.uint8 if fp8 else dt))
    g.update({k: gb.t for k, gb in guards.items()})
    te.te_layernorm_mlp_bwd(inp["dy"], inp["x"], inp["gamma"], inp["w1"], inp["w2"], g["h"],
                            g["ln"], g["mu"], g["rs"], g["dx"], g["dgamma"], g["dw1"], g["dw2"],
                            dbeta=g["dbeta"], dbias1=g["db1"], dbias2=g["db2"],
                            saved_dh=g["dh"], **kw)
    for k, gb in guards.items():
        gb.check(k)
    if inp["norm"] != "layernorm":  # no shift: the gradient of the unused beta is zero
        assert int(g["dbeta"].count_nonzero().item()) == 0
        g["dbeta"] = None
    return g


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
    check_mlp_bwd(inp, g, fp8)
    if fp8:  # delayed scaling: the given scales are used as they are
        assert g["qs"].grad.scale.item() == SCALES["grad"]


@pytest.mark.parametrize("name,shape", CASES)
def test_mlp_backward_fp8_current_scaling(name, shape):
    """Every quantizer in current scaling: the forward's casts and the backward's dH cast each
    take a separate amax pass (the dbias reduction runs in dH's amax pass).  Each scale must be
    the recipe's function of the GPU's amax; the weights' amaxes come from identical inputs and
    must be identical; dH's amax is held by the step check."""
    inp = _inputs(name, shape)
    g = run_gpu(inp, True, mode="current")
    qs = g["qs"]
    for name_q, q in (("x", qs.x), ("act", qs.act), ("grad", qs.grad), ("kernel1", qs.kernel1)):
        amax = np.float32(q.amax.item())
        assert np.float32(q.scale.item()) == nx.compute_scale(amax)[0], name_q
    w1 = nx.bf16_round(np64(inp["w1"]))
    assert np.float32(qs.kernel1.amax.item()) == nx.amax_of(w1)
    check_mlp_bwd(inp, g, True)


@pytest.mark.parametrize("act", ["geglu", "reglu"])
@pytest.mark.parametrize("fp8", [False, True])
def test_mlp_backward_other_gated(act, fp8):
    """("gelu", "linear") and ("relu", "linear"): the recomputed activation, the gated
    dact + dbias (+ E4M3) step and the rest of the backward."""
    inp = _inputs("llama_rms_mlp", dict(M=256, H=512, F=528))
    inp["act"] = act
    g = run_gpu(inp, fp8)
    check_mlp_bwd(inp, g, fp8)


def _cols(t, idx):
    """Columns idx of a device tensor, on the host as float64 (E4M3: the codes)."""
    sel = t[:, torch.as_tensor(idx, device=t.device)]
    return codes(sel) if t.dtype == torch.uint8 else np64(sel)


def _decoded_rows_matmul(t, b, chunk=2048):
    """decode(t) @ b and |decode(t)| @ |b| for an E4M3 (or bf16) device tensor t, in row chunks
    so that the float64 copy of t never exists whole on the host."""
    out, absout = [], []
    for r0 in range(0, t.shape[0], chunk):
        part = t[r0:r0 + chunk]
        v = decode(codes(part)) if t.dtype == torch.uint8 else np64(part)
        out.append(v @ b)
        absout.append(np.abs(v) @ np.abs(b))
    return np.concatenate(out), np.concatenate(absout)


@pytest.mark.parametrize("fp8", [False, True])
def test_mlp_backward_full_size_sampled(fp8):
    """The full GPT backward (16384 tokens, 4096 -> 16384 -> 4096, gelu), bf16 and with dH in
    E4M3 (delayed scaling), in the launch configuration the benchmark times.  The oracle's steps
    run from the backward's inputs on a sample: all of dbias2, rows of dx (row-local), columns f
    of the hidden layer (dH[:, f], dbias1[f], dW1[:, f], dW2[f, :]) and columns of dgamma and
    dbeta (which need dln over every token)."""
    inp = make_inputs("gpt_ln_mlp_bwd", device=DEV)
    g = run_gpu(inp, fp8)
    for k in ("dx", "dgamma", "dbeta", "dw1", "dw2", "db1", "db2"):
        assert torch.isfinite(g[k].float()).all(), k
    M, H, F = inp["M"], inp["H"], inp["F"]
    qs = g["qs"]
    rng = np.random.default_rng(11)
    rows = np.sort(rng.choice(M, 8, replace=False))
    rows[-1] = M - 1
    feats = np.sort(rng.choice(F, 6, replace=False))
    feats[-1] = F - 1
    hcols = np.sort(rng.choice(H, 6, replace=False))
    f64 = lambda k: np64(inp[k])
    dy, x, gamma, w1, w2 = f64("dy"), f64("x"), f64("gamma"), f64("w1"), f64("w2")
    mu, rs = np64(g["mu"]), np64(g["rs"])
    assert_in_window(g["db2"], ob.colsum(dy), 0.0, "dbias2")
    # columns f of the hidden layer
    h_c = _cols(g["h"], feats)                                     # [M, 6]
    a64 = ob.act_fwd(h_c, "gelu")
    J_a = bf16_jump(a64, ACT_REL * np.abs(a64))
    a = nx.bf16_round(a64)
    dw2, w_dw2 = gemm_ref(a.T, dy)
    assert_in_window(np64(g["dw2"])[feats], dw2, w_dw2 + J_a.T @ np.abs(dy), "dW2 rows",
                     stored="bf16")
    w2b = nx.bf16_round(w2)
    da64, w_da = gemm_ref(dy, w2b[feats].T)                        # [M, 6]
    g_scale = np.float32(qs.grad.scale.item()) if fp8 else None
    dh_c = _cols(g["dh"], feats)
    check_dact(dh_c if fp8 else dh_c.astype(np.float64), np64(g["db1"])[feats], da64, w_da,
               h_c, "gelu", q_scale=g_scale, what="dH columns")
    if fp8:
        dh_cv = decode(dh_c)
        ln_v = decode(codes(g["ln"]))
        a_w1 = float(np.float32(qs.x.scale_inv.item()) * np.float32(qs.grad.scale_inv.item()))
        w1q = decode(quantize_fast(w1, np.float32(qs.kernel1.scale.item())))
        a_dln = float(np.float32(qs.grad.scale_inv.item()) * np.float32(qs.kernel1.scale_inv.item()))
        # the amax of dH covers at least the sampled columns' values
        pre_max = np.abs(nx.to_f32(ob.act_bwd(nx.bf16_round(da64), h_c, "gelu"))).max()
        assert qs.grad.amax.item() >= pre_max * (1 - 1e-4)
    else:
        dh_cv, ln_v = dh_c, np64(g["ln"])
        w1q, a_w1, a_dln = nx.bf16_round(w1), 1.0, 1.0
    dw1, w_dw1 = gemm_ref(ln_v.T, dh_cv, a_w1)                     # [H, 6]
    assert_in_window(np64(g["dw1"])[:, feats], dw1, w_dw1, "dW1 columns", stored="bf16")
    # rows of dx: dln of those rows from the GPU's dH
    dh_r = g["dh"][torch.as_tensor(rows, device=DEV)]
    dh_rv = decode(codes(dh_r)) if fp8 else np64(dh_r)
    dln_r, w_dln_r = gemm_ref(dh_rv, w1q.T, a_dln)
    check_norm_dx(np64(g["dx"])[rows], dln_r, w_dln_r, x[rows], mu[rows], rs[rows], gamma,
                  "layernorm", False, what="dx rows")
    # columns of dgamma / dbeta: dln[:, hcols] over every token
    dln_c, abs_c = _decoded_rows_matmul(g["dh"], w1q[hcols].T)
    dln_c = dln_c * a_dln
    w_dln_c = ACC_REL * abs(a_dln) * abs_c + SCALE_REL * np.abs(dln_c)
    check_norm_params(np64(g["dgamma"])[hcols], np64(g["dbeta"])[hcols], dln_c, w_dln_c,
                      x[:, hcols], mu, rs, "layernorm", what="norm columns")
