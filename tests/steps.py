"""Step-by-step parity of the backward passes, given identical inputs.

A backward call's inputs are dy, x, gamma, the kernels and what the forward saved (h, the
normalized output, mu, rsigma).  The checks below take the oracle's primitives (act_fwd,
act_bwd, gemm, colsum, norm_bwd) in the order of ``oracle.block.*_bwd_from_saved``, from
exactly those tensors, so that every comparison holds a step of the chain
to the pages' tight rules -- fp32 reductions to 1e-4, E4M3 codes and amax exact up to the
rounding of the step's own fp32 arithmetic -- and adds only what the rounding of an fp32
intermediate inside the chain can explain (the windows of ``parity``):

* a bf16 GEMM output (da, dln, and the weight gradients) may land on either bf16 neighbour
  where its exact value lies within the fp32 accumulation window of a rounding midpoint;
* the activation and its gradient carry the kernels' fp32 arithmetic error (ACT_REL);
* a consumer that is linear in such an intermediate (dH in da, dbias1 in dH, dx / dgamma /
  dbeta in dln) inherits the intermediate's jumps through the absolute values of its
  coefficients.

Where the GPU exposes an intermediate (dH through ``saved_dh``), the next step starts from the
GPU's tensor, so that its check does not carry the window of the step before.
"""

from __future__ import annotations

import numpy as np

from oracle import block as ob
from oracle import numerics as nx
from parity import (assert_e4m3_codes, assert_in_window, bf16_jump, codes, gemm_window, np64)

ACT_REL = 1e-5   # fp32 error of the kernels' activation and activation-gradient values, relative
NORM_REL = 1e-5  # fp32 error of the norm backward's per-element arithmetic, relative
SCALE_REL = 2.0 ** -22  # the fp32 product of two dequantization factors, relative


def stored_values(t, scale_inv=None):
    """float64 values a GEMM reads from a stored tensor: decoded E4M3 codes (with the factor
    returned separately) or the bf16 / fp32 numbers."""
    if scale_inv is None:
        return np64(t)
    return nx.e4m3_decode(codes(t))


def gemm_ref(a, b, alpha=1.0):
    """Float64 alpha * a @ b and its window (fp32 accumulation + the factor's rounding)."""
    v = ob.gemm(a, b, None, alpha)
    return v, gemm_window(a, b, alpha) + SCALE_REL * np.abs(v)


def xhat_of(x, mu, rs, norm):
    return (x - mu[:, None]) * rs[:, None] if norm == "layernorm" else x * rs[:, None]


def xhat_err(x, mu, rs, norm):
    """Absolute fp32 error window of xhat = x rs - mu rs (a cancellation when |mu| >> std)."""
    m = np.abs(mu)[:, None] if norm == "layernorm" else 0.0
    return NORM_REL * (np.abs(x) + m) * rs[:, None]


def _stored_dln(dln64, w_dln, dln_dtype):
    """The upstream gradient as the norm backward reads it, and how far the GPU's copy may sit
    from it: a bf16 GEMM output may be one bf16 step away wherever dln64 +- w_dln straddles a
    midpoint; an input given in fp32 (or bf16) is identical on both sides."""
    if dln_dtype == "gemm_bf16":
        return nx.bf16_round(dln64), bf16_jump(dln64, w_dln)
    return np.asarray(dln64, np.float64), np.zeros(np.shape(dln64))


def check_norm_dx(g_dx, dln64, w_dln, x, mu, rs, gamma, norm, zc, what="dx", stored="bf16",
                  dln_dtype="gemm_bf16"):
    """dx of whole rows against the oracle's norm backward of the upstream gradient (see
    _stored_dln), stored as ``stored``."""
    dln, J = _stored_dln(dln64, w_dln, dln_dtype)
    dx, _, _ = ob.norm_bwd(dln, x, mu, rs, gamma, norm, zc)
    g = ob.applied_gain(gamma, zc)[None, :]
    xh = xhat_of(x, mu, rs, norm)
    aJ = J * np.abs(g)
    w_dx = aJ + np.abs(xh) * (aJ * np.abs(xh)).mean(axis=1, keepdims=True)
    d = dln * g
    proj = (d * xh).mean(axis=1, keepdims=True)
    mag = np.abs(d) + np.abs(xh) * np.abs(proj)
    if norm == "layernorm":
        w_dx = w_dx + aJ.mean(axis=1, keepdims=True)
        mag = mag + np.abs(d.mean(axis=1, keepdims=True))
    # xhat is formed in fp32 from x, mu and rsigma: its absolute error enters through both
    # places it appears
    xe = xhat_err(x, mu, rs, norm)
    w_dx = w_dx + xe * np.abs(proj) + np.abs(xh) * (np.abs(d) * xe).mean(axis=1, keepdims=True)
    w_dx = rs[:, None] * (w_dx + NORM_REL * mag)
    if stored == "bf16":
        assert_in_window(g_dx, dx, w_dx, what, stored="bf16")
    else:  # fp32 storage: the window plus one fp32 rounding
        got = np64(g_dx)
        bad = np.abs(got - dx) > w_dx + 2.0 ** -23 * np.abs(dx)
        assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outside the window"


def check_norm_params(g_dgamma, g_dbeta, dln64, w_dln, x, mu, rs, norm, what="norm",
                      dln_dtype="gemm_bf16"):
    """dgamma = sum_i dln * xhat and dbeta = sum_i dln over all rows, for the columns given
    (x, dln64, w_dln hold those columns of every row)."""
    dln, J = _stored_dln(dln64, w_dln, dln_dtype)
    xh = xhat_of(x, mu, rs, norm)
    xerr = xhat_err(x, mu, rs, norm)
    assert_in_window(g_dgamma, (dln * xh).sum(axis=0),
                     (J * np.abs(xh)).sum(axis=0) + (np.abs(dln) * xerr).sum(axis=0),
                     f"{what} dgamma")
    if norm == "layernorm" and g_dbeta is not None:
        assert_in_window(g_dbeta, dln.sum(axis=0), J.sum(axis=0), f"{what} dbeta")


def _deriv_terms(z, base):
    """Sum of the absolute values of the terms a kernel adds to form base'(z): near a root of
    the derivative (gelu' at about -0.75, silu' at about -1.28) the terms cancel, so their fp32
    rounding is relative to this sum, not to the result."""
    z = np.asarray(z, np.float64)
    if base == "gelu":
        t = np.tanh(ob.SQRT_2_OVER_PI * (z + ob.GELU_CUBIC * z ** 3))
        return (0.5 * (1 + t) + np.abs(0.5 * z * (1 - t * t) * ob.SQRT_2_OVER_PI
                                       * (1 + 3 * ob.GELU_CUBIC * z * z)))
    if base == "silu":
        sg = 1.0 / (1.0 + np.exp(-z))
        return sg + np.abs(z * sg * (1 - sg))
    return np.zeros_like(z)  # relu: exact


def dact_terms(da, h, act):
    """A bound on the magnitude of the terms behind da * act'(h), per element of dH (the
    linear half of a gated pair is one product, bounded by its own value)."""
    da, h = np.abs(np.asarray(da, np.float64)), np.asarray(h, np.float64)
    if act in ob.GATE_BASE:
        F = h.shape[1] // 2
        g, lin = h[:, :F], h[:, F:]
        return np.concatenate([da * np.abs(lin) * _deriv_terms(g, ob.GATE_BASE[act]),
                               np.zeros_like(lin)], axis=1)
    return da * _deriv_terms(h, act)


def check_dact(g_dh, g_db1, da64, w_da, h, act, q_scale=None, g_amax=None, what="dH"):
    """dH = da * act'(h) and its column sums, given the oracle's da (whose bf16 rounding may
    differ from the GPU's where da64 +- w_da straddles a midpoint) and the GPU's own h.
    ``q_scale`` = the fp32 scale dH was cast with (FP8), else dH is bf16."""
    J_da = bf16_jump(da64, w_da)
    da = nx.bf16_round(da64)
    pre = nx.to_f32(ob.act_bwd(da, h, act))
    w = ACT_REL * (np.abs(pre) + dact_terms(da, h, act)) + np.abs(ob.act_bwd(J_da, h, act))
    if g_db1 is not None:
        assert_in_window(g_db1, ob.colsum(pre), w.sum(axis=0), f"{what} dbias")
    if q_scale is None:
        assert_in_window(g_dh, pre, w, what, stored="bf16")
        return
    assert_e4m3_codes(g_dh, nx.quantize(pre, q_scale), pre32=pre, scale=q_scale, rel=0.0,
                      abs_tol=w, max_frac=2e-3, what=f"{what} e4m3")
    if g_amax is not None:
        lo = float(np.max(np.abs(pre) - w))
        hi = float(np.max(np.abs(pre) + w))
        assert lo * (1 - 2.0 ** -23) <= g_amax <= hi * (1 + 2.0 ** -23), (
            f"{what} amax {g_amax} outside [{lo}, {hi}]")


def check_mlp_bwd(inp, gpu, fp8):
    """Every output of te_layernorm_mlp_bwd, step by step, at small sizes (all elements).

    ``gpu`` holds the forward's saved tensors (h, ln, mu, rs), the backward's outputs, the
    saved dH and the quantizer set."""
    f = lambda k: np64(inp[k])
    dy, x, gamma, w1, w2 = f("dy"), f("x"), f("gamma"), f("w1"), f("w2")
    act, norm, zc = inp["act"], inp["norm"], inp["zero_centered_gamma"]
    M = dy.shape[0]
    qs = gpu["qs"]
    h = np64(gpu["h"])
    mu, rs = np64(gpu["mu"]), np64(gpu["rs"])
    # dbias2: column sums of dy (identical input)
    assert_in_window(gpu["db2"], ob.colsum(dy), 0.0, "dbias2")
    # dW2 = a^T dy, a = bf16(act(h)) recomputed from the GPU's h
    a64 = ob.act_fwd(h, act)
    J_a = bf16_jump(a64, ACT_REL * np.abs(a64))
    a = nx.bf16_round(a64)
    dw2, w_dw2 = gemm_ref(a.T, dy)
    assert_in_window(gpu["dw2"], dw2, w_dw2 + J_a.T @ np.abs(dy), "dW2", stored="bf16")
    # da = dy W2^T, then dH and dbias1
    w2b = nx.bf16_round(w2)
    da64, w_da = gemm_ref(dy, w2b.T)
    g_scale = np.float32(qs.grad.scale.item()) if fp8 else None
    check_dact(gpu["dh"], gpu["db1"], da64, w_da, h, act, q_scale=g_scale,
               g_amax=qs.grad.amax.item() if fp8 else None)
    if fp8:
        assert np.float32(qs.grad.scale_inv.item()) == np.float32(1.0) / g_scale
    # dW1 = ln^T dH and dln = dH W1^T from the GPU's own ln and dH
    if fp8:
        ln = stored_values(gpu["ln"], 1)
        dh = stored_values(gpu["dh"], 1)
        w1q = nx.e4m3_decode(nx.quantize(nx.bf16_round(w1), np.float32(qs.kernel1.scale.item())))
        a_w1 = float(np.float32(qs.x.scale_inv.item()) * np.float32(qs.grad.scale_inv.item()))
        a_dln = float(np.float32(qs.grad.scale_inv.item()) * np.float32(qs.kernel1.scale_inv.item()))
    else:
        ln, dh, w1q, a_w1, a_dln = np64(gpu["ln"]), np64(gpu["dh"]), nx.bf16_round(w1), 1.0, 1.0
    dw1, w_dw1 = gemm_ref(ln.T, dh, a_w1)
    assert_in_window(gpu["dw1"], dw1, w_dw1, "dW1", stored="bf16")
    dln64, w_dln = gemm_ref(dh, w1q.T, a_dln)
    check_norm_dx(gpu["dx"], dln64, w_dln, x, mu, rs, gamma, norm, zc)
    check_norm_params(gpu["dgamma"], gpu.get("dbeta"), dln64, w_dln, x, mu, rs, norm)
    assert M == dh.shape[0]


def check_dense_bwd(dy, x, gamma, kernel, gpu, fp8, norm, zc):
    """Every output of te_layernorm_dense_bwd, step by step (all elements), from the backward's
    inputs: dy, x, gamma, the kernel and the forward's saved ln, mu, rsigma.  In FP8 mode dy and
    the kernel are cast from identical inputs, so their codes are the oracle's exactly."""
    qs = gpu["qs"]
    mu, rs = np64(gpu["mu"]), np64(gpu["rs"])
    assert_in_window(gpu["dbias"], ob.colsum(dy), 0.0, "dbias")
    if fp8:
        s_g = np.float32(qs.grad.scale.item())
        s_k = np.float32(qs.kernel1.scale.item())
        gy = nx.e4m3_decode(nx.quantize(dy, s_g))
        kq = nx.e4m3_decode(nx.quantize(kernel, s_k))
        ln = stored_values(gpu["ln"], 1)
        a_dk = float(np.float32(qs.x.scale_inv.item()) * np.float32(qs.grad.scale_inv.item()))
        a_dln = float(np.float32(qs.grad.scale_inv.item()) * np.float32(qs.kernel1.scale_inv.item()))
    else:
        gy, kq, ln, a_dk, a_dln = dy, kernel, np64(gpu["ln"]), 1.0, 1.0
    dk, w_dk = gemm_ref(ln.T, gy, a_dk)
    assert_in_window(gpu["dkernel"], dk, w_dk, "dkernel", stored="bf16")
    dln64, w_dln = gemm_ref(gy, kq.T, a_dln)
    check_norm_dx(gpu["dx"], dln64, w_dln, x, mu, rs, gamma, norm, zc)
    check_norm_params(gpu["dgamma"], gpu.get("dbeta"), dln64, w_dln, x, mu, rs, norm)
