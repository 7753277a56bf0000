"""Seeded synthetic inputs for the fused norm + feed-forward block.

This module only draws random tensors; it holds none of the block's arithmetic.  Both the
CPU oracle's tests and the CUDA path's tests and benchmark take their inputs from here, so the
two sides always see the same bytes.

Every workload draws fp32 numbers from one ``torch.Generator`` seeded with ``seed`` on the
requested device, in the order listed for it below, and rounds them once (round to nearest
even) to the workload's storage dtype.  The same seed on a different device gives different
numbers, so a test draws on one device and hands the same tensors to both sides.

Workloads (shapes at full size; every one can be drawn smaller by overriding M/H/F/N):

* ``tiny_ln_mlp``   LayerNorm-MLP forward in fp32: x[64,128] ~ N(0,1), gamma = 1 + N(0,0.1),
  beta ~ N(0,0.1), W1[128,512], W2[512,128] ~ N(0,0.02), b1, b2 ~ N(0,0.02); layernorm,
  eps 1e-6, gelu (tanh form), no quantization.
* ``qkv_ln_dense``  LayerNorm -> Dense (QKV projection), bf16 and E4M3: x[16384,8192] ~ N(0,1)
  with every row r where r % 100 == 0 (1% of rows) multiplied by 8; kernel[8192,24576] ~
  N(0,0.01); bias ~ N(0,0.02); gamma = 1 + N(0,0.1); beta ~ N(0,0.1); eps 1e-5.
* ``gpt_ln_mlp``    GPT-style LayerNorm-MLP forward, gelu: tokens 16384, hidden 4096, ffn 16384;
  x ~ N(0,1); W1[4096,16384], W2[16384,4096] ~ N(0,0.02); b1, b2 ~ N(0,0.02); gamma, beta
  drawn as in ``qkv_ln_dense``; eps 1e-6.
* ``llama_rms_mlp`` Llama-style RMSNorm-MLP forward, gated SwiGLU ("silu", "linear"), no
  biases, zero-centered gamma: tokens 8192, hidden 4096, ffn 14336; x ~ N(0,1);
  W1[4096, 2*14336], W2[14336,4096] ~ N(0,0.02); gamma ~ N(0,0.05); eps 1e-6.
* ``gpt_ln_mlp_bwd`` the ``gpt_ln_mlp`` tensors followed by the upstream gradient
  dY[16384,4096] ~ N(0,1).
"""

from __future__ import annotations

import torch

WORKLOADS = {
    "tiny_ln_mlp": dict(M=64, H=128, F=512, norm="layernorm", act="gelu", eps=1e-6,
                        dtype="f32", gated=False, has_bias=True, zero_centered_gamma=False),
    "qkv_ln_dense": dict(M=16384, H=8192, N=24576, norm="layernorm", eps=1e-5,
                         dtype="bf16", has_bias=True, zero_centered_gamma=False),
    "gpt_ln_mlp": dict(M=16384, H=4096, F=16384, norm="layernorm", act="gelu", eps=1e-6,
                       dtype="bf16", gated=False, has_bias=True, zero_centered_gamma=False),
    "llama_rms_mlp": dict(M=8192, H=4096, F=14336, norm="rmsnorm", act="swiglu", eps=1e-6,
                          dtype="bf16", gated=True, has_bias=False, zero_centered_gamma=True),
    "gpt_ln_mlp_bwd": dict(M=16384, H=4096, F=16384, norm="layernorm", act="gelu", eps=1e-6,
                           dtype="bf16", gated=False, has_bias=True, zero_centered_gamma=False),
}

_TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def _normal(gen, shape, std, device, mean=0.0):
    t = torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t


def make_inputs(name: str, device="cpu", seed: int = 0, **shape) -> dict:
    """Draw the tensors of workload ``name`` (see the module docstring).

    ``shape`` may override M, H, F or N.  Returns a dict of tensors in the workload's storage
    dtype together with the scalar settings (``eps``, ``norm``, ``act`` ...).
    """
    cfg = dict(WORKLOADS[name])
    cfg.update({k: v for k, v in shape.items() if v is not None})
    dt = _TORCH_DTYPE[cfg["dtype"]]
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    M, H = cfg["M"], cfg["H"]
    out = dict(cfg)
    out["name"] = name
    if name == "tiny_ln_mlp":
        F = cfg["F"]
        out["x"] = _normal(gen, (M, H), 1.0, device)
        out["gamma"] = _normal(gen, (H,), 0.1, device, mean=1.0)
        out["beta"] = _normal(gen, (H,), 0.1, device)
        out["w1"] = _normal(gen, (H, F), 0.02, device)
        out["w2"] = _normal(gen, (F, H), 0.02, device)
        out["b1"] = _normal(gen, (F,), 0.02, device)
        out["b2"] = _normal(gen, (H,), 0.02, device)
    elif name == "qkv_ln_dense":
        N = cfg["N"]
        x = _normal(gen, (M, H), 1.0, device)
        x[0::100] *= 8.0
        out["x"] = x
        out["kernel"] = _normal(gen, (H, N), 0.01, device)
        out["bias"] = _normal(gen, (N,), 0.02, device)
        out["gamma"] = _normal(gen, (H,), 0.1, device, mean=1.0)
        out["beta"] = _normal(gen, (H,), 0.1, device)
    elif name in ("gpt_ln_mlp", "gpt_ln_mlp_bwd"):
        F = cfg["F"]
        out["x"] = _normal(gen, (M, H), 1.0, device)
        out["w1"] = _normal(gen, (H, F), 0.02, device)
        out["w2"] = _normal(gen, (F, H), 0.02, device)
        out["b1"] = _normal(gen, (F,), 0.02, device)
        out["b2"] = _normal(gen, (H,), 0.02, device)
        out["gamma"] = _normal(gen, (H,), 0.1, device, mean=1.0)
        out["beta"] = _normal(gen, (H,), 0.1, device)
        if name == "gpt_ln_mlp_bwd":
            out["dy"] = _normal(gen, (M, H), 1.0, device)
    elif name == "llama_rms_mlp":
        F = cfg["F"]
        out["x"] = _normal(gen, (M, H), 1.0, device)
        out["w1"] = _normal(gen, (H, 2 * F), 0.02, device)
        out["w2"] = _normal(gen, (F, H), 0.02, device)
        out["gamma"] = _normal(gen, (H,), 0.05, device)
        # RMSNorm ignores beta; the block's signature still carries one.
        out["beta"] = torch.zeros(H, device=device)
    else:
        raise KeyError(name)
    for k in ("x", "gamma", "beta", "w1", "w2", "b1", "b2", "kernel", "bias", "dy"):
        if k in out:
            out[k] = out[k].to(dt).contiguous()
    return out


def random_tensor(shape, std=1.0, device="cpu", seed=0, dtype="bf16", mean=0.0):
    """One N(mean, std) tensor of ``shape`` rounded to ``dtype`` (kernel-level parity cases)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return _normal(gen, shape, std, device, mean=mean).to(_TORCH_DTYPE[dtype]).contiguous()
