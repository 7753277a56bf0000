"""The fused norm + feed-forward block, written out plainly in float64.

Test infrastructure, never product code (see ``oracle/__init__.py``).

Sources (TransformerEngine JAX pages):

* "LayerNorm MLP" page, Description: the forward pass is (1) normalization, (2) first GEMM
  with bias, (3) activation, (4) second GEMM with bias; the backward pass uses one fused
  operation for activation gradient + bias reduction + quantization and produces gradients
  for all parameters.  Signature / I/O Contract: ``norm_type`` is "layernorm" or "rmsnorm",
  ``zero_centered_gamma``, ``epsilon`` (default 1e-6), ``kernels=[kernel1, kernel2]``,
  ``biases=[bias1, bias2]`` (either may be None), ``activation_type`` (default ("relu",)).
* "LayerNorm Dense" page, Description: normalization, then the normalized output and the
  kernel are quantized, then one GEMM with optional bias; output = LayerNorm(x) @ kernel + bias.
* "Activation" page, Description and I/O Contract: activations such as ("gelu",) and the gated
  pair ("silu", "linear"); with a quantizer the output is quantized and dequantized back.

Where the pages say nothing the readings are:

* LayerNorm uses the population (biased) variance, with epsilon inside the square root.
  RMSNorm divides by sqrt(mean(x^2) + eps) and has no shift (beta is accepted and unused).
  ``zero_centered_gamma`` means the applied gain is 1 + gamma.
* "gelu" is the tanh form 0.5 h (1 + tanh(sqrt(2/pi) (h + 0.044715 h^3))).
* The gated pair ("silu", "linear") splits GEMM1's 2F output columns as [gate | linear]:
  columns [0, F) go through silu, columns [F, 2F) are the linear factor.
* GEMM1's output plus bias is rounded to the activation dtype before the activation (the
  unfused four-step pipeline materializes it there); that rounded tensor is what is saved for
  the backward.
* FP8: E4M3 with one scale per tensor (see ``numerics``).  A GEMM on E4M3 operands multiplies
  the decoded codes, then scales the sum by scale_inv_a * scale_inv_b and adds the bias.
* The bias gradient is reduced from the unquantized fp32 activation gradient.

All sums are float64; a value is rounded only where the block stores it.
"""

from __future__ import annotations

import math

import numpy as np
from scipy.special import expit

from .numerics import (amax_of, bf16_round, compute_scale, dequantize, e4m3_decode,
                       quantize, to_f32)

SQRT_2_OVER_PI = math.sqrt(2.0 / math.pi)
GELU_CUBIC = 0.044715

# ----------------------------------------------------------------------------------------
# Normalization (LayerNorm MLP page, Description step (1); LayerNorm Dense page, Description)
# ----------------------------------------------------------------------------------------


def applied_gain(gamma, zero_centered_gamma: bool) -> np.ndarray:
    g = np.asarray(gamma, dtype=np.float64)
    return 1.0 + g if zero_centered_gamma else g


def norm_fwd(x, gamma, beta, norm_type: str, zero_centered_gamma: bool, eps: float):
    """Row-wise LayerNorm or RMSNorm of x[M, H].  Returns (y, mu, rsigma), all float64.

    layernorm: mu = mean(x), var = mean((x - mu)^2), rsigma = 1 / sqrt(var + eps),
               y = (x - mu) * rsigma * g + beta
    rmsnorm:   rsigma = 1 / sqrt(mean(x^2) + eps), y = x * rsigma * g; mu is reported as 0.
    g = gamma, or 1 + gamma with zero_centered_gamma.
    """
    x = np.asarray(x, dtype=np.float64)
    g = applied_gain(gamma, zero_centered_gamma)
    if norm_type == "layernorm":
        mu = x.mean(axis=1)
        var = ((x - mu[:, None]) ** 2).mean(axis=1)
        rs = 1.0 / np.sqrt(var + eps)
        y = (x - mu[:, None]) * rs[:, None] * g[None, :] + np.asarray(beta, np.float64)[None, :]
    elif norm_type == "rmsnorm":
        mu = np.zeros(x.shape[0])
        rs = 1.0 / np.sqrt((x * x).mean(axis=1) + eps)
        y = x * rs[:, None] * g[None, :]
    else:
        raise ValueError(norm_type)
    return y, mu, rs


def norm_bwd(dy, x, mu, rsigma, gamma, norm_type: str, zero_centered_gamma: bool):
    """Gradients of the normalization for upstream dy[M, H].  Returns (dx, dgamma, dbeta).

    With xhat = (x - mu) * rsigma (layernorm) or x * rsigma (rmsnorm) and dxhat = dy * g:
      layernorm: dx = rsigma * (dxhat - mean(dxhat) - xhat * mean(dxhat * xhat))
      rmsnorm:   dx = rsigma * (dxhat - xhat * mean(dxhat * xhat))
      dgamma = sum over rows of dy * xhat (the same for a zero-centered gamma, since
      d(1 + gamma)/dgamma = 1); dbeta = sum over rows of dy (layernorm only; None for rmsnorm).
    """
    dy = np.asarray(dy, dtype=np.float64)
    x = np.asarray(x, dtype=np.float64)
    rs = np.asarray(rsigma, dtype=np.float64)[:, None]
    g = applied_gain(gamma, zero_centered_gamma)[None, :]
    if norm_type == "layernorm":
        xhat = (x - np.asarray(mu, np.float64)[:, None]) * rs
    else:
        xhat = x * rs
    dxhat = dy * g
    proj = (dxhat * xhat).mean(axis=1, keepdims=True)
    if norm_type == "layernorm":
        dx = rs * (dxhat - dxhat.mean(axis=1, keepdims=True) - xhat * proj)
        dbeta = dy.sum(axis=0)
    else:
        dx = rs * (dxhat - xhat * proj)
        dbeta = None
    dgamma = (dy * xhat).sum(axis=0)
    return dx, dgamma, dbeta


# ----------------------------------------------------------------------------------------
# Activations (Activation page: Overview, I/O Contract, Usage Examples)
# ----------------------------------------------------------------------------------------


def relu(h):
    return np.maximum(h, 0.0)


def _half_one_plus_tanh(u):
    """0.5 (1 + tanh(u)), evaluated as the logistic function of 2u (the same number: 1 + tanh(u)
    = 2 / (1 + exp(-2u))), which keeps its relative accuracy where 1 + tanh(u) would cancel
    (u below about -5, where float64 tanh(u) rounds to within a few ulps of -1)."""
    return expit(2.0 * np.asarray(u, dtype=np.float64))


def gelu(h):
    """Tanh-form GELU 0.5 h (1 + tanh(sqrt(2/pi) (h + 0.044715 h^3)))."""
    h = np.asarray(h, dtype=np.float64)
    return h * _half_one_plus_tanh(SQRT_2_OVER_PI * (h + GELU_CUBIC * h ** 3))


def silu(z):
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def d_relu(h):
    """relu'(h) = 1 for h > 0, else 0 (0 at h == 0)."""
    return (np.asarray(h) > 0).astype(np.float64)


def d_gelu(h):
    """Derivative of the tanh-form gelu: with u = sqrt(2/pi)(h + 0.044715 h^3), t = tanh(u),
    gelu' = 0.5 (1 + t) + 0.5 h (1 - t^2) sqrt(2/pi) (1 + 3 * 0.044715 h^2).
    0.5 (1 + t) and 1 - t^2 = 4 * [0.5 (1 + t)] * [0.5 (1 - t)] are taken through the logistic
    function (see _half_one_plus_tanh), so neither cancels in the tails."""
    h = np.asarray(h, dtype=np.float64)
    u = SQRT_2_OVER_PI * (h + GELU_CUBIC * h ** 3)
    p, m = _half_one_plus_tanh(u), _half_one_plus_tanh(-u)
    return p + 2.0 * h * p * m * SQRT_2_OVER_PI * (1.0 + 3.0 * GELU_CUBIC * h * h)


def d_silu(z):
    """silu'(z) = s (1 + z (1 - s)) with s = 1 / (1 + exp(-z))."""
    z = np.asarray(z, dtype=np.float64)
    s = 1.0 / (1.0 + np.exp(-z))
    return s * (1.0 + z * (1.0 - s))


# Gated pairs (Activation page, Usage Examples / activation_type tuples): (base, "linear")
GATE_BASE = {"swiglu": "silu", "geglu": "gelu", "reglu": "relu"}
GATED = {"swiglu": True, "geglu": True, "reglu": True, "relu": False, "gelu": False,
         "silu": False}
_BASE_FWD = {"relu": relu, "gelu": gelu, "silu": silu}
_BASE_BWD = {"relu": d_relu, "gelu": d_gelu, "silu": d_silu}


def act_fwd(h, act: str):
    """Activation of h[M, N_in].  A gated type (base, "linear") -- "swiglu" = ("silu",
    "linear"), "geglu" = ("gelu", "linear"), "reglu" = ("relu", "linear") -- has N_in = 2F: the
    first F columns are the gate, the last F the linear factor; output base(gate) * linear
    [M, F]."""
    h = np.asarray(h, dtype=np.float64)
    if act in _BASE_FWD:
        return _BASE_FWD[act](h)
    if act in GATE_BASE:
        F = h.shape[1] // 2
        return _BASE_FWD[GATE_BASE[act]](h[:, :F]) * h[:, F:]
    raise ValueError(act)


def act_bwd(da, h, act: str):
    """Gradient w.r.t. the activation input h, given da = dL/d(act output).

    Gated: d_gate = da * linear * base'(gate), d_linear = da * base(gate), concatenated
    [d_gate | d_linear] like h.
    """
    da = np.asarray(da, dtype=np.float64)
    h = np.asarray(h, dtype=np.float64)
    if act in _BASE_BWD:
        return da * _BASE_BWD[act](h)
    if act in GATE_BASE:
        F = h.shape[1] // 2
        g, lin = h[:, :F], h[:, F:]
        base = GATE_BASE[act]
        return np.concatenate([da * lin * _BASE_BWD[base](g), da * _BASE_FWD[base](g)], axis=1)
    raise ValueError(act)


# ----------------------------------------------------------------------------------------
# Storage: how a float64 result becomes the stored tensor
# ----------------------------------------------------------------------------------------


class Stored:
    """A stored tensor: its values as float64, plus E4M3 codes / amax when quantized.

    ``value`` is what a consumer reads: the fp32 or bf16 number, or for E4M3 the decoded code
    (the consumer applies ``scale_inv``).  ``pre`` is the fp32 number before the cast, and
    ``amax`` the max |pre| (computed for every dtype).
    """

    def __init__(self, v64, dtype: str, scale=None):
        self.dtype = dtype
        self.pre = to_f32(v64)
        self.amax = amax_of(self.pre)
        self.codes = None
        self.scale = None
        self.scale_inv = None
        if dtype == "f32":
            self.value = self.pre
        elif dtype == "bf16":
            self.value = bf16_round(self.pre)
        elif dtype == "e4m3":
            if scale is None:  # current scaling: this tensor's own amax
                scale, _ = compute_scale(self.amax)
            self.scale = np.float32(scale)
            self.scale_inv = np.float32(1.0) / self.scale
            self.codes = quantize(self.pre, self.scale)
            self.value = e4m3_decode(self.codes)
        else:
            raise ValueError(dtype)

    def dequantized(self):
        if self.dtype != "e4m3":
            return self.value
        return dequantize(self.codes, self.scale_inv)

    def inv(self) -> float:
        return 1.0 if self.scale_inv is None else float(self.scale_inv)


# ----------------------------------------------------------------------------------------
# GEMM with bias (LayerNorm MLP page, Description steps (2), (4))
# ----------------------------------------------------------------------------------------


def gemm(a, b, bias=None, alpha=1.0):
    """alpha * (a @ b) + bias in float64; a[M, K], b[K, N], bias[N] or None."""
    out = np.asarray(a, np.float64) @ np.asarray(b, np.float64)
    out = out * float(alpha)
    if bias is not None:
        out = out + np.asarray(bias, np.float64)[None, :]
    return out


def gemm_alpha(sa, sb) -> float:
    """The fp32 dequantization factor scale_inv_a * scale_inv_b applied to an FP8 GEMM sum."""
    return float(np.float32(sa) * np.float32(sb))


def colsum(v):
    """Column sums over all rows (the bias gradient reduction), float64."""
    return np.asarray(v, dtype=np.float64).sum(axis=0)


# ----------------------------------------------------------------------------------------
# Composed forward passes
# ----------------------------------------------------------------------------------------


def _f64(t):
    if t is None:
        return None
    if hasattr(t, "detach"):
        return t.detach().cpu().double().numpy()
    return np.asarray(t, dtype=np.float64)


def layernorm_dense_fwd(x, kernel, gamma, beta, bias, norm_type="layernorm",
                        zero_centered_gamma=False, eps=1e-6, dtype="bf16", fp8=None):
    """LayerNorm Dense page: y = norm(x) @ kernel + bias, optionally through FP8.

    ``fp8`` = None (no quantization) or a dict with the fp32 scales ``x`` and ``kernel`` (None
    for a scale taken from the tensor's own amax).  Returns a dict of every stored tensor.
    """
    x, kernel, gamma, beta, bias = map(_f64, (x, kernel, gamma, beta, bias))
    y, mu, rs = norm_fwd(x, gamma, beta, norm_type, zero_centered_gamma, eps)
    if fp8 is None:
        ln = Stored(y, dtype)
        w = Stored(kernel, dtype)
        out = gemm(ln.value, w.value, bias)
    else:
        ln = Stored(y, "e4m3", fp8.get("x"))
        w = Stored(kernel, "e4m3", fp8.get("kernel"))
        out = gemm(ln.value, w.value, bias, gemm_alpha(ln.scale_inv, w.scale_inv))
    return dict(ln=ln, mu=mu, rsigma=rs, kernel=w, out=Stored(out, dtype))


def layernorm_mlp_fwd(x, gamma, beta, w1, w2, b1, b2, norm_type="layernorm",
                      zero_centered_gamma=False, eps=1e-6, act="gelu", dtype="bf16", fp8=None):
    """LayerNorm MLP page, forward steps (1)-(4).

    ``dtype`` is the activation/storage dtype ("bf16" or "f32").  ``fp8`` = None or a dict of
    fp32 scales for ``x`` (normalized output), ``w1``, ``act`` (activation output) and ``w2``;
    a missing or None entry means the tensor's own amax sets its scale.
    Returns every stored intermediate: ln, mu, rsigma, h (GEMM1 + bias, rounded to ``dtype``),
    a (activation output), out.
    """
    x, gamma, beta, w1, w2, b1, b2 = map(_f64, (x, gamma, beta, w1, w2, b1, b2))
    y, mu, rs = norm_fwd(x, gamma, beta, norm_type, zero_centered_gamma, eps)
    q = fp8 is not None
    ln = Stored(y, "e4m3", fp8.get("x")) if q else Stored(y, dtype)
    W1 = Stored(w1, "e4m3", fp8.get("w1")) if q else Stored(w1, dtype)
    h = Stored(gemm(ln.value, W1.value, b1, gemm_alpha(ln.inv(), W1.inv())), dtype)
    a64 = act_fwd(h.value, act)
    a = Stored(a64, "e4m3", fp8.get("act")) if q else Stored(a64, dtype)
    W2 = Stored(w2, "e4m3", fp8.get("w2")) if q else Stored(w2, dtype)
    out = Stored(gemm(a.value, W2.value, b2, gemm_alpha(a.inv(), W2.inv())), dtype)
    return dict(ln=ln, mu=mu, rsigma=rs, w1=W1, h=h, a=a, w2=W2, out=out)


def layernorm_mlp_bwd(dy, x, gamma, beta, w1, w2, b1, b2, norm_type="layernorm",
                      zero_centered_gamma=False, eps=1e-6, act="gelu", dtype="bf16",
                      fp8=None):
    """Backward of ``layernorm_mlp_fwd`` (LayerNorm MLP page, Description, backward pass):
    the forward pass, then ``layernorm_mlp_bwd_from_saved`` on what it saves.

    ``fp8`` = None or a dict of fp32 scales ``x``, ``w1``, ``act``, ``w2`` (forward) and ``grad``
    (dh); None entries take the tensor's own amax.  Returns the backward's dict plus ``fwd``.
    """
    fwd = layernorm_mlp_fwd(x, gamma, beta, w1, w2, b1, b2, norm_type, zero_centered_gamma,
                            eps, act, dtype, fp8=None if fp8 is None else
                            {k: fp8.get(k) for k in ("x", "w1", "act", "w2")})
    ln = fwd["ln"]
    res = layernorm_mlp_bwd_from_saved(dy, x, gamma, w1, w2, fwd["h"].value, ln.value, ln.inv(),
                                       fwd["mu"], fwd["rsigma"], norm_type, zero_centered_gamma,
                                       act, dtype, fp8)
    res["fwd"] = fwd
    return res


def layernorm_mlp_bwd_from_saved(dy, x, gamma, w1, w2, h, ln, ln_scale_inv, mu, rsigma,
                                 norm_type="layernorm", zero_centered_gamma=False, act="gelu",
                                 dtype="bf16", fp8=None):
    """The MLP backward given what the forward saved (LayerNorm MLP page, Description, backward
    pass): h = GEMM1 output + bias (the activation input), ln = the normalized output as stored
    (decoded E4M3 codes, dequantized by ``ln_scale_inv``, or ``dtype`` values), mu, rsigma.

    Order: db2 = colsum(dy); a = act(h) recomputed; dW2 = a^T dy; da = dy W2^T;
    dh = da * act'(h) (fp32), db1 = colsum(dh), dh stored (E4M3 with its own scale when
    ``fp8`` is given, else ``dtype``); dln = dh W1^T; dW1 = ln^T dh; then the norm backward
    gives dx, dgamma, dbeta.  In FP8 mode only dh, ln and W1 are E4M3 operands (W1 cast with
    ``fp8["w1"]``, dh with ``fp8["grad"]``; None = the tensor's own amax); dy, W2 and the
    recomputed activation stay in ``dtype``.
    """
    dy, h, ln = _f64(dy), _f64(h), _f64(ln)
    xs, g = _f64(x), _f64(gamma)
    db2 = colsum(dy)
    a_re = Stored(act_fwd(h, act), dtype)
    dW2 = Stored(gemm(a_re.value.T, dy), dtype)
    w2s = Stored(_f64(w2), dtype)
    da = Stored(gemm(dy, w2s.value.T), dtype)
    dh64 = act_bwd(da.value, h, act)
    dh32 = to_f32(dh64)
    db1 = colsum(dh32)
    if fp8 is None:
        dh = Stored(dh32, dtype)
        w1s = Stored(_f64(w1), dtype)
        dln = Stored(gemm(dh.value, w1s.value.T), dtype)
        dW1 = Stored(gemm(ln.T, dh.value), dtype)
    else:
        dh = Stored(dh32, "e4m3", fp8.get("grad"))
        w1q = Stored(_f64(w1), "e4m3", fp8.get("w1"))
        dln = Stored(gemm(dh.value, w1q.value.T, None, gemm_alpha(dh.scale_inv, w1q.scale_inv)),
                     dtype)
        dW1 = Stored(gemm(ln.T, dh.value, None, gemm_alpha(ln_scale_inv, dh.scale_inv)), dtype)
    dx, dgamma, dbeta = norm_bwd(dln.value, xs, mu, rsigma, g, norm_type, zero_centered_gamma)
    return dict(db2=db2, a_re=a_re, dW2=dW2, da=da, dh=dh, db1=db1, dln=dln, dW1=dW1,
                dx=Stored(dx, dtype), dgamma=dgamma, dbeta=dbeta)


def layernorm_dense_bwd(dy, x, gamma, beta, kernel, bias, norm_type="layernorm",
                        zero_centered_gamma=False, eps=1e-6, dtype="bf16", fp8=None):
    """Backward of ``layernorm_dense_fwd``: the forward pass, then
    ``layernorm_dense_bwd_from_saved`` on what it saves.  ``fp8`` = None or a dict of fp32
    scales ``x``, ``kernel`` and ``grad`` (None: the tensor's own amax).  Returns the
    backward's dict plus ``fwd``."""
    fwd = layernorm_dense_fwd(x, kernel, gamma, beta, bias, norm_type, zero_centered_gamma, eps,
                              dtype, fp8=None if fp8 is None else
                              {k: fp8.get(k) for k in ("x", "kernel")})
    ln = fwd["ln"]
    res = layernorm_dense_bwd_from_saved(dy, x, gamma, kernel, ln.value, ln.inv(), fwd["mu"],
                                         fwd["rsigma"], norm_type, zero_centered_gamma, dtype,
                                         fp8)
    res["fwd"] = fwd
    return res


def layernorm_dense_bwd_from_saved(dy, x, gamma, kernel, ln, ln_scale_inv, mu, rsigma,
                                   norm_type="layernorm", zero_centered_gamma=False,
                                   dtype="bf16", fp8=None):
    """The LayerNorm Dense backward given what the forward saved (LayerNorm Dense page,
    Description: the gradients of x, the kernel, gamma, beta and the bias, with FP8
    intermediate gradients): ln = the normalized output as stored (decoded E4M3 codes,
    dequantized by ``ln_scale_inv``, or ``dtype`` values), mu, rsigma.

    Order: dbias = colsum(dy) over the unquantized dy; dy is the GEMM operand (E4M3 with the
    ``grad`` scale, or its own amax, when ``fp8`` is given; else ``dtype``); dln = dy kernel^T;
    dkernel = ln^T dy; then the norm backward gives dx, dgamma, dbeta.  In FP8 mode the GEMM
    operands are dy, ln and the kernel (cast with ``fp8["kernel"]``), all E4M3.
    """
    dy, ln = _f64(dy), _f64(ln)
    xs, g = _f64(x), _f64(gamma)
    dbias = colsum(dy)
    if fp8 is None:
        gy = Stored(dy, dtype)
        ks = Stored(_f64(kernel), dtype)
        dln = Stored(gemm(gy.value, ks.value.T), dtype)
        dk = Stored(gemm(ln.T, gy.value), dtype)
    else:
        gy = Stored(dy, "e4m3", fp8.get("grad"))
        kq = Stored(_f64(kernel), "e4m3", fp8.get("kernel"))
        dln = Stored(gemm(gy.value, kq.value.T, None, gemm_alpha(gy.scale_inv, kq.scale_inv)),
                     dtype)
        dk = Stored(gemm(ln.T, gy.value, None, gemm_alpha(ln_scale_inv, gy.scale_inv)), dtype)
    dx, dgamma, dbeta = norm_bwd(dln.value, xs, mu, rsigma, g, norm_type, zero_centered_gamma)
    return dict(dbias=dbias, dy=gy, dln=dln, dkernel=dk, dx=Stored(dx, dtype), dgamma=dgamma,
                dbeta=dbeta)
