"""Pins for the oracle's block arithmetic (oracle/block.py), against things other than itself.

* Normalization: torch.nn.functional.layer_norm / rms_norm in float64 (library routines), the
  closed forms of a normalized row (zero mean, mean square var / (var + eps)), the scale
  identity LN(c x; eps) = LN(x; eps / c^2), a constant row, zero-centered gamma.
* Norm backward: torch.autograd through the float64 library norms, and central differences.
* Activations: the exact erf-form GELU (scipy) that the tanh form approximates, logistic silu
  (scipy's expit), odd-part identities, SwiGLU with a unit linear half.
* Activation gradients: central finite differences of the forward.
* GEMM and the bias reduction: brute-force loops on tiny shapes.
* The composed forward and backward: finite differences through the whole tiny block, and an
  FP8 forward rebuilt from torch's float8_e4m3fn conversion.
"""

import numpy as np
import pytest
import scipy.special as sp
import torch
import torch.nn.functional as F

from oracle import block as ob
from oracle import numerics as nx


def rng(seed=0):
    return np.random.default_rng(seed)


# ------------------------------- normalization -------------------------------------------


@pytest.mark.parametrize("M,H", [(1, 8), (7, 136), (33, 512)])
@pytest.mark.parametrize("zc", [False, True])
def test_layernorm_matches_torch(M, H, zc):
    r = rng(M + H)
    x = r.normal(size=(M, H)) * 3 + 1
    g = r.normal(size=H) * 0.1 + (0 if zc else 1)
    b = r.normal(size=H) * 0.1
    y, mu, rs = ob.norm_fwd(x, g, b, "layernorm", zc, 1e-5)
    w = torch.tensor(1 + g if zc else g)
    ref = F.layer_norm(torch.tensor(x), (H,), w, torch.tensor(b), eps=1e-5).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(mu, x.mean(1), rtol=1e-13)
    np.testing.assert_allclose(rs, 1 / np.sqrt(x.var(1) + 1e-5), rtol=1e-13)


@pytest.mark.parametrize("zc", [False, True])
def test_rmsnorm_matches_torch(zc):
    r = rng(3)
    x = r.normal(size=(17, 264))
    g = r.normal(size=264) * 0.05
    y, mu, rs = ob.norm_fwd(x, g, np.zeros(264) + 7.0, "rmsnorm", zc, 1e-6)
    w = torch.tensor(1 + g if zc else g)
    ref = F.rms_norm(torch.tensor(x), (264,), w, eps=1e-6).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    assert np.all(mu == 0)


def test_norm_closed_forms():
    r = rng(4)
    x = r.normal(size=(50, 128)) * r.uniform(0.01, 10, size=(50, 1))
    eps = 1e-3
    y, _, _ = ob.norm_fwd(x, np.ones(128), np.zeros(128), "layernorm", False, eps)
    var = x.var(1)
    np.testing.assert_allclose(y.mean(1), 0, atol=1e-12)
    np.testing.assert_allclose((y ** 2).mean(1), var / (var + eps), rtol=1e-12)
    y, _, _ = ob.norm_fwd(x, np.ones(128), np.zeros(128), "rmsnorm", False, eps)
    ms = (x ** 2).mean(1)
    np.testing.assert_allclose((y ** 2).mean(1), ms / (ms + eps), rtol=1e-12)


def test_norm_scale_identity_and_constant_row():
    r = rng(5)
    x = r.normal(size=(4, 64))
    g, b = r.normal(size=64), r.normal(size=64)
    for c in (8.0, 0.25):
        y1, _, _ = ob.norm_fwd(c * x, g, b, "layernorm", False, 1e-5)
        y2, _, _ = ob.norm_fwd(x, g, b, "layernorm", False, 1e-5 / c ** 2)
        np.testing.assert_allclose(y1, y2, rtol=1e-12, atol=1e-12)
    const = np.full((2, 64), 3.25)
    y, _, _ = ob.norm_fwd(const, g, b, "layernorm", False, 1e-6)
    np.testing.assert_allclose(y, np.broadcast_to(b, y.shape), atol=1e-12)


def test_zero_centered_gamma_is_one_plus_gamma():
    r = rng(6)
    x, g, b = r.normal(size=(5, 32)), r.normal(size=32) * 0.1, r.normal(size=32)
    for nt in ("layernorm", "rmsnorm"):
        a, _, _ = ob.norm_fwd(x, g, b, nt, True, 1e-6)
        c, _, _ = ob.norm_fwd(x, 1 + g, b, nt, False, 1e-6)
        np.testing.assert_allclose(a, c, rtol=1e-14)


@pytest.mark.parametrize("nt", ["layernorm", "rmsnorm"])
@pytest.mark.parametrize("zc", [False, True])
def test_norm_bwd_matches_autograd(nt, zc):
    r = rng(7)
    M, H = 6, 40
    x = r.normal(size=(M, H)) * 2
    g = r.normal(size=H) * 0.1 + (0 if zc else 1)
    b = r.normal(size=H) * 0.1
    dy = r.normal(size=(M, H))
    _, mu, rs = ob.norm_fwd(x, g, b, nt, zc, 1e-5)
    dx, dg, db = ob.norm_bwd(dy, x, mu, rs, g, nt, zc)
    xt = torch.tensor(x, requires_grad=True)
    gt = torch.tensor(g, requires_grad=True)
    bt = torch.tensor(b, requires_grad=True)
    w = 1 + gt if zc else gt
    if nt == "layernorm":
        y = F.layer_norm(xt, (H,), w, bt, eps=1e-5)
    else:
        y = F.rms_norm(xt, (H,), w, eps=1e-5)
    y.backward(torch.tensor(dy))
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dg, gt.grad.numpy(), rtol=1e-10, atol=1e-12)
    if nt == "layernorm":
        np.testing.assert_allclose(db, bt.grad.numpy(), rtol=1e-12, atol=1e-12)
    else:
        assert db is None


def test_norm_bwd_finite_differences():
    r = rng(8)
    x = r.normal(size=(3, 12))
    g, b = r.normal(size=12), r.normal(size=12)
    G = r.normal(size=(3, 12))
    loss = lambda xx: (ob.norm_fwd(xx, g, b, "layernorm", False, 1e-5)[0] * G).sum()
    _, mu, rs = ob.norm_fwd(x, g, b, "layernorm", False, 1e-5)
    dx, _, _ = ob.norm_bwd(G, x, mu, rs, g, "layernorm", False)
    h = 1e-6
    fd = np.zeros_like(x)
    for i in range(x.shape[0]):
        for j in range(x.shape[1]):
            e = np.zeros_like(x)
            e[i, j] = h
            fd[i, j] = (loss(x + e) - loss(x - e)) / (2 * h)
    np.testing.assert_allclose(dx, fd, rtol=1e-6, atol=1e-8)


# ------------------------------- activations ---------------------------------------------


def test_gelu_tanh_form_close_to_erf_form():
    x = np.linspace(-8, 8, 20001)
    exact = x * 0.5 * (1 + sp.erf(x / np.sqrt(2)))
    err = np.abs(ob.gelu(x) - exact)
    # the tanh form differs from x*Phi(x) by under 5e-4 everywhere (about 4.7e-4 at |x| ~ 2)
    assert err.max() < 5e-4
    assert err.max() > 1e-5  # and it is the tanh form, not the exact one


@pytest.mark.parametrize("h", [-12.0, -9.5, -6.875, -4.0, -1.5, -0.75, -1e-3, 0.0, 2e-3, 0.5,
                               1.0, 3.0, 6.875, 11.0])
def test_gelu_and_derivative_against_high_precision(h):
    """The tanh form and its derivative evaluated with 200 significant digits (mpmath) from the
    definition as written, 0.5 h (1 + tanh(u)): the oracle keeps 1e-13 relative accuracy in the
    far tails, where a float64 evaluation of 1 + tanh(u) itself would cancel."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 200
    hm = mp.mpf(h)
    c = mp.sqrt(2 / mp.pi)
    u = c * (hm + mp.mpf("0.044715") * hm ** 3)
    t = mp.tanh(u)
    g = hm / 2 * (1 + t)
    dg = (1 + t) / 2 + hm / 2 * (1 - t * t) * c * (1 + 3 * mp.mpf("0.044715") * hm * hm)
    assert ob.gelu(np.array([h]))[0] == pytest.approx(float(g), rel=1e-13, abs=1e-300)
    assert ob.d_gelu(np.array([h]))[0] == pytest.approx(float(dg), rel=1e-12, abs=1e-300)


def test_activation_identities():
    x = np.linspace(-10, 10, 4001)
    np.testing.assert_allclose(ob.gelu(x) - ob.gelu(-x), x, atol=1e-12)
    np.testing.assert_allclose(ob.silu(x) - ob.silu(-x), x, atol=1e-12)
    np.testing.assert_allclose(ob.silu(x), x * sp.expit(x), rtol=1e-13, atol=1e-15)
    assert ob.gelu(np.array([0.0]))[0] == 0.0
    np.testing.assert_array_equal(ob.relu(x), np.where(x > 0, x, 0.0))
    gate = rng(9).normal(size=(5, 8))
    h = np.concatenate([gate, np.ones_like(gate)], axis=1)
    np.testing.assert_allclose(ob.act_fwd(h, "swiglu"), ob.silu(gate), rtol=1e-15)
    lin = rng(10).normal(size=(5, 8))
    h = np.concatenate([gate, lin], axis=1)
    np.testing.assert_allclose(ob.act_fwd(h, "swiglu"), gate * sp.expit(gate) * lin, rtol=1e-13)
    # ("gelu", "linear") and ("relu", "linear"): the gate half goes through the base function
    h1 = np.concatenate([gate, np.ones_like(gate)], axis=1)
    np.testing.assert_allclose(ob.act_fwd(h1, "geglu"), ob.gelu(gate), rtol=1e-15)
    np.testing.assert_array_equal(ob.act_fwd(h, "reglu"), np.maximum(gate, 0.0) * lin)
    swapped = np.concatenate([lin, gate], axis=1)
    assert not np.allclose(ob.act_fwd(swapped, "geglu"), ob.act_fwd(h, "geglu"))


@pytest.mark.parametrize("act", ["gelu", "silu", "relu", "swiglu", "geglu", "reglu"])
def test_act_bwd_finite_differences(act):
    r = rng(11)
    h = r.normal(size=(4, 16)) * 2
    h[np.abs(h) < 1e-3] = 0.5  # keep away from relu's kink
    n_out = 8 if ob.GATED[act] else 16
    da = r.normal(size=(4, n_out))
    got = ob.act_bwd(da, h, act)
    step = 1e-6
    fd = np.zeros_like(h)
    for i in range(h.shape[0]):
        for j in range(h.shape[1]):
            e = np.zeros_like(h)
            e[i, j] = step
            fd[i, j] = ((ob.act_fwd(h + e, act) - ob.act_fwd(h - e, act)) * da).sum() / (2 * step)
    np.testing.assert_allclose(got, fd, rtol=1e-6, atol=1e-8)


def test_gelu_derivative_limits():
    assert ob.d_gelu(np.array([0.0]))[0] == 0.5
    np.testing.assert_allclose(ob.d_gelu(np.array([12.0, -12.0])), [1.0, 0.0], atol=1e-12)
    assert ob.d_relu(np.array([0.0]))[0] == 0.0


# ------------------------------- GEMM and reductions -------------------------------------


def test_gemm_brute_force():
    r = rng(12)
    a, b, bias = r.normal(size=(3, 5)), r.normal(size=(5, 4)), r.normal(size=4)
    want = np.zeros((3, 4))
    for i in range(3):
        for j in range(4):
            acc = 0.0
            for k in range(5):
                acc += a[i, k] * b[k, j]
            want[i, j] = 0.5 * acc + bias[j]
    np.testing.assert_allclose(ob.gemm(a, b, bias, alpha=0.5), want, rtol=1e-14)
    np.testing.assert_allclose(ob.gemm(a, b), a @ b, rtol=1e-14)


def test_colsum_brute_force():
    v = rng(13).normal(size=(9, 6))
    want = [sum(v[i, j] for i in range(9)) for j in range(6)]
    np.testing.assert_allclose(ob.colsum(v), want, rtol=1e-14)


# ------------------------------- composition ---------------------------------------------


def _tiny_block(seed=14, gated=False):
    r = rng(seed)
    M, H, Fd = 3, 8, 6
    x = r.normal(size=(M, H))
    g = 1 + 0.1 * r.normal(size=H)
    b = 0.1 * r.normal(size=H)
    w1 = 0.3 * r.normal(size=(H, 2 * Fd if gated else Fd))
    w2 = 0.3 * r.normal(size=(Fd, H))
    b1 = 0.1 * r.normal(size=w1.shape[1])
    b2 = 0.1 * r.normal(size=H)
    return x, g, b, w1, w2, b1, b2


def _plain_forward(x, g, b, w1, w2, b1, b2, act, nt="layernorm"):
    y, _, _ = ob.norm_fwd(x, g, b, nt, False, 1e-5)
    return ob.act_fwd(y @ w1 + b1, act) @ w2 + b2


@pytest.mark.parametrize("act,nt", [("gelu", "layernorm"), ("swiglu", "rmsnorm"),
                                    ("relu", "layernorm"), ("geglu", "layernorm"),
                                    ("reglu", "rmsnorm")])
def test_block_bwd_finite_differences(act, nt):
    """Every gradient of the composed backward against central differences of the forward.

    dtype f32 keeps the oracle's storage rounding at fp32, far below the FD tolerance."""
    x, g, b, w1, w2, b1, b2 = _tiny_block(gated=ob.GATED[act])
    if act in ("relu", "reglu"):
        w1 = w1 + 0.0
    G = rng(15).normal(size=(x.shape[0], w2.shape[1]))
    res = ob.layernorm_mlp_bwd(G, x, g, b, w1, w2, b1, b2, nt, False, 1e-5, act, "f32")
    params = dict(x=x, g=g, b=b, w1=w1, w2=w2, b1=b1, b2=b2)
    grads = dict(x=res["dx"].value, g=res["dgamma"], b=res["dbeta"], w1=res["dW1"].value,
                 w2=res["dW2"].value, b1=res["db1"], b2=res["db2"])
    step = 1e-6
    for name, p in params.items():
        if nt == "rmsnorm" and name == "b":
            assert grads["b"] is None
            continue
        fd = np.zeros_like(p)
        for idx in np.ndindex(p.shape):
            pp, pm = dict(params), dict(params)
            pp[name] = p.copy()
            pm[name] = p.copy()
            pp[name][idx] += step
            pm[name][idx] -= step
            fd[idx] = ((_plain_forward(**pp, act=act, nt=nt) - _plain_forward(**pm, act=act, nt=nt))
                       * G).sum() / (2 * step)
        np.testing.assert_allclose(grads[name], fd, rtol=2e-5, atol=2e-6, err_msg=name)


def test_forward_matches_plain_composition():
    x, g, b, w1, w2, b1, b2 = _tiny_block(seed=16)
    res = ob.layernorm_mlp_fwd(x, g, b, w1, w2, b1, b2, "layernorm", False, 1e-5, "gelu", "f32")
    want = _plain_forward(x, g, b, w1, w2, b1, b2, "gelu")
    np.testing.assert_allclose(res["out"].value, want, rtol=1e-5, atol=1e-6)


def _torch_fake_quant(v, scale):
    """fp32(v * scale) -> float8_e4m3fn (torch's conversion) -> float64 decoded codes."""
    t = torch.tensor(v, dtype=torch.float32) * torch.tensor(scale, dtype=torch.float32)
    t = t.clamp(-448, 448)  # torch's conversion does not saturate; the recipe does
    return t.to(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_fp8_forward_matches_torch_float8_composition():
    """The FP8 forward rebuilt with torch's float8 conversion and fp64 matmul, with fixed
    scales (so the torch version needs no amax logic)."""
    r = rng(17)
    M, H, Fd = 16, 32, 48
    x = r.normal(size=(M, H)).astype(np.float32).astype(np.float64)
    g = 1 + 0.1 * r.normal(size=H)
    b = 0.1 * r.normal(size=H)
    w1 = 0.02 * r.normal(size=(H, Fd))
    w2 = 0.02 * r.normal(size=(Fd, H))
    b1, b2 = 0.02 * r.normal(size=Fd), 0.02 * r.normal(size=H)
    s = dict(x=np.float32(64.0), w1=np.float32(4096.0), act=np.float32(256.0), w2=np.float32(8192.0))
    res = ob.layernorm_mlp_fwd(x, g, b, w1, w2, b1, b2, "layernorm", False, 1e-6, "gelu",
                               "bf16", fp8=s)
    y, _, _ = ob.norm_fwd(x, g, b, "layernorm", False, 1e-6)
    qx = _torch_fake_quant(nx.to_f32(y), s["x"])
    qw1 = _torch_fake_quant(w1, s["w1"])
    alpha1 = float(np.float32(1 / s["x"]) * np.float32(1 / s["w1"]))
    h = torch.tensor(qx @ qw1 * alpha1 + b1, dtype=torch.float32).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(res["ln"].value, qx)
    np.testing.assert_array_equal(res["h"].value, h)
    a = _torch_fake_quant(nx.to_f32(ob.gelu(h)), s["act"])
    np.testing.assert_array_equal(res["a"].value, a)
    qw2 = _torch_fake_quant(w2, s["w2"])
    alpha2 = float(np.float32(1 / s["act"]) * np.float32(1 / s["w2"]))
    out = torch.tensor(a @ qw2 * alpha2 + b2, dtype=torch.float32).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(res["out"].value, out)


def test_fp8_current_scaling_uses_own_amax():
    r = rng(18)
    v = r.normal(size=(8, 16)) * 3
    st = ob.Stored(v, "e4m3")
    s, si = nx.compute_scale(nx.amax_of(nx.to_f32(v)))
    assert st.scale == s and st.scale_inv == si
    assert np.abs(st.dequantized()).max() == pytest.approx(float(st.amax), rel=1e-6)


@pytest.mark.parametrize("nt,zc", [("layernorm", False), ("rmsnorm", True)])
def test_dense_bwd_finite_differences(nt, zc):
    """LayerNorm Dense backward: every gradient against central differences of the plain
    forward norm(x) @ kernel + bias (dtype f32 keeps the storage rounding far below the FD
    tolerance)."""
    r = rng(31)
    M, H, N = 5, 8, 6
    x = r.normal(size=(M, H)) + 0.3
    g = (0.1 if zc else 1.0) * r.normal(size=H) * 0.3 + (0.0 if zc else 1.0)
    b = 0.1 * r.normal(size=H)
    k = 0.3 * r.normal(size=(H, N))
    bias = 0.1 * r.normal(size=N)
    G = r.normal(size=(M, N))
    res = ob.layernorm_dense_bwd(G, x, g, b, k, bias, nt, zc, 1e-5, "f32")

    def fwd(x, g, b, k, bias):
        y, _, _ = ob.norm_fwd(x, g, b, nt, zc, 1e-5)
        return y @ k + bias

    params = dict(x=x, g=g, b=b, k=k, bias=bias)
    grads = dict(x=res["dx"].value, g=res["dgamma"], b=res["dbeta"], k=res["dkernel"].value,
                 bias=res["dbias"])
    step = 1e-6
    for name, p in params.items():
        if nt == "rmsnorm" and name == "b":
            assert grads["b"] is None
            continue
        fd = np.zeros_like(p)
        for idx in np.ndindex(p.shape):
            pp, pm = dict(params), dict(params)
            pp[name] = p.copy()
            pm[name] = p.copy()
            pp[name][idx] += step
            pm[name][idx] -= step
            fd[idx] = ((fwd(**pp) - fwd(**pm)) * G).sum() / (2 * step)
        np.testing.assert_allclose(grads[name], fd, rtol=2e-5, atol=2e-6, err_msg=name)


def test_fp8_dense_bwd_matches_torch_float8_composition():
    """The FP8 LayerNorm Dense backward GEMMs rebuilt with torch's float8 conversion and fp64
    matmul, with fixed scales: dln = q(dy) q(kernel)^T and dkernel = q(ln)^T q(dy), each scaled
    by the product of the two dequantization factors and rounded to bf16."""
    r = rng(32)
    M, H, N = 16, 32, 48
    x = r.normal(size=(M, H)).astype(np.float32).astype(np.float64)
    g = 1 + 0.1 * r.normal(size=H)
    b = 0.1 * r.normal(size=H)
    k = 0.02 * r.normal(size=(H, N))
    dy = nx.bf16_round(r.normal(size=(M, N)))
    s = dict(x=np.float32(64.0), kernel=np.float32(4096.0), grad=np.float32(32.0))
    res = ob.layernorm_dense_bwd(dy, x, g, b, k, None, "layernorm", False, 1e-6, "bf16", fp8=s)
    y, _, _ = ob.norm_fwd(x, g, b, "layernorm", False, 1e-6)
    qx = _torch_fake_quant(nx.to_f32(y), s["x"])
    qk = _torch_fake_quant(k, s["kernel"])
    qdy = _torch_fake_quant(dy, s["grad"])
    bf = lambda v: torch.tensor(v, dtype=torch.float32).to(torch.bfloat16).double().numpy()
    a1 = float(np.float32(1 / s["grad"]) * np.float32(1 / s["kernel"]))
    a2 = float(np.float32(1 / s["x"]) * np.float32(1 / s["grad"]))
    np.testing.assert_array_equal(res["dy"].value, qdy)
    np.testing.assert_array_equal(res["dln"].value, bf(qdy @ qk.T * a1))
    np.testing.assert_array_equal(res["dkernel"].value, bf(qx.T @ qdy * a2))
    np.testing.assert_allclose(res["dbias"], dy.sum(axis=0), rtol=1e-12)


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_fp8_mlp_bwd_matches_torch_float8_composition(act):
    """The FP8 branch of the MLP backward rebuilt from torch: float8_e4m3fn conversion for the
    quantized operands, autograd through torch's tanh-form gelu / silu for the activation
    gradient and through torch's layer_norm for the norm backward, fp64 matmul for the GEMMs,
    all with fixed scales.  It fixes which tensor each step reads: dbias1 sums the unquantized
    fp32 dH; dH is cast with the grad scale alone; dln = q(dH) q(W1)^T and dW1 = q(ln)^T q(dH),
    each scaled by the product of its two operands' dequantization factors; dW2 and da use the
    bf16 recomputed activation, dy and bf16 W2."""
    r = rng(33)
    M, H, Fd = 16, 32, 24
    gated = ob.GATED[act]
    F1 = 2 * Fd if gated else Fd
    x = r.normal(size=(M, H)).astype(np.float32).astype(np.float64)
    g = 1 + 0.1 * r.normal(size=H)
    b = 0.1 * r.normal(size=H)
    w1 = nx.bf16_round(0.05 * r.normal(size=(H, F1)))
    w2 = nx.bf16_round(0.05 * r.normal(size=(Fd, H)))
    b1 = nx.bf16_round(0.02 * r.normal(size=F1))
    dy = nx.bf16_round(r.normal(size=(M, H)))
    s = dict(x=np.float32(32.0), w1=np.float32(2048.0), act=np.float32(16.0),
             w2=np.float32(2048.0), grad=np.float32(256.0))
    res = ob.layernorm_mlp_bwd(dy, x, g, b, w1, w2, b1, None, "layernorm", False, 1e-6, act,
                               "bf16", fp8=s)
    bf = lambda v: torch.tensor(v, dtype=torch.float32).to(torch.bfloat16).double().numpy()
    inv = lambda k: float(np.float32(1) / s[k])
    # forward operands: E4M3 normalized output and W1, bf16 GEMM1 output
    xt = torch.tensor(x, requires_grad=True)
    gt = torch.tensor(g, requires_grad=True)
    bt = torch.tensor(b, requires_grad=True)
    y = F.layer_norm(xt, (H,), gt, bt, eps=1e-6)
    qx = _torch_fake_quant(nx.to_f32(y.detach().numpy()), s["x"])
    qw1 = _torch_fake_quant(w1, s["w1"])
    h = bf(qx @ qw1 * float(np.float32(inv("x")) * np.float32(inv("w1"))) + b1)
    np.testing.assert_array_equal(res["fwd"]["h"].value, h)

    def act_t(ht):
        if not gated:
            return F.gelu(ht, approximate="tanh")
        return F.silu(ht[:, :Fd]) * ht[:, Fd:]

    ht = torch.tensor(h, requires_grad=True)
    a = act_t(ht)
    a_re = bf(a.detach().numpy())
    np.testing.assert_array_equal(res["a_re"].value, a_re)
    np.testing.assert_array_equal(res["dW2"].value, bf(a_re.T @ dy))
    da = bf(dy @ w2.T)
    np.testing.assert_array_equal(res["da"].value, da)
    a.backward(torch.tensor(da))
    dh32 = nx.to_f32(ht.grad.numpy())
    np.testing.assert_allclose(res["db1"], dh32.sum(axis=0), rtol=1e-12, atol=1e-12)
    qdh = _torch_fake_quant(dh32, s["grad"])
    np.testing.assert_array_equal(res["dh"].value, qdh)
    assert res["dh"].scale == s["grad"]
    dln = bf(qdh @ qw1.T * float(np.float32(inv("grad")) * np.float32(inv("w1"))))
    np.testing.assert_array_equal(res["dln"].value, dln)
    dw1 = bf(qx.T @ qdh * float(np.float32(inv("x")) * np.float32(inv("grad"))))
    np.testing.assert_array_equal(res["dW1"].value, dw1)
    y.backward(torch.tensor(dln))
    np.testing.assert_allclose(res["dx"].value, bf(xt.grad.numpy()), rtol=2.0 ** -8, atol=1e-12)
    np.testing.assert_allclose(res["dgamma"], gt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(res["dbeta"], bt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(res["db2"], dy.sum(axis=0), rtol=1e-12)
