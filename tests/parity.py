"""Comparison rules between the CUDA path and the oracle.

* GEMM outputs (contraction K): max |gpu - ref| <= 2e-2 * sqrt(K) * rms(A) * rms(B), i.e. a
  2e-2 fraction of the output's expected magnitude.
* Elementwise bf16 outputs: |gpu - ref| <= 2e-2 * |ref| + 1e-3 * rms(ref).
* fp32 reductions (mu, rsigma, dbias, dgamma, dbeta): |gpu - ref| <= 1e-4 * max(|ref|, rms(ref)).
* E4M3 codes from identical fp32 inputs: bit-exact.  Codes of values the GPU computed itself
  (through a norm or a GEMM epilogue): equal, except at most one step apart on at most 0.1% of
  elements, and only where the oracle's pre-cast value lies within ``near`` (relative) of a
  rounding boundary, so that fp32 evaluation-order differences can explain the flip.
"""

from __future__ import annotations

import math

import numpy as np
import torch

from oracle import numerics as nx


def np64(t) -> np.ndarray:
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return t.detach().cpu().view(torch.uint8).numpy().astype(np.int64)
    return t.detach().cpu().double().numpy()


def codes(t) -> np.ndarray:
    return t.detach().cpu().view(torch.uint8).numpy().astype(np.int64)


def rms(v) -> float:
    v = np.asarray(v, dtype=np.float64)
    return float(np.sqrt(np.mean(v * v))) if v.size else 0.0


def assert_gemm_close(got, ref, K, rms_a, rms_b, what="gemm"):
    got, ref = np64(got), np.asarray(ref, np.float64)
    tol = 2e-2 * math.sqrt(K) * rms_a * rms_b
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    worst = float(err.max()) if err.size else 0.0
    assert worst <= tol, f"{what}: max err {worst:.3e} > tol {tol:.3e} (K={K})"
    return worst / tol if tol else 0.0


def assert_elementwise_close(got, ref, what="elementwise", rel=2e-2, abs_rms=1e-3):
    got, ref = np64(got), np.asarray(ref, np.float64)
    tol = rel * np.abs(ref) + abs_rms * rms(ref)
    bad = np.abs(got - ref) > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                           f"first got {got[bad][:4]} ref {ref[bad][:4]}")


def assert_reduction_close(got, ref, what="reduction", rel=1e-4):
    got, ref = np64(got), np.asarray(ref, np.float64)
    scale = np.maximum(np.abs(ref), rms(ref))
    err = np.abs(got - ref)
    bad = err > rel * scale
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} out of tolerance; worst "
                           f"{float((err / scale).max()):.3e}")


def e4m3_step(c: np.ndarray) -> np.ndarray:
    """Signed position of each code on the ordered E4M3 grid (so a one-step flip differs by 1)."""
    c = np.asarray(c, np.int64)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def assert_e4m3_codes(got, want_codes, pre32=None, scale=None, near=1e-5, max_frac=1e-3,
                      what="e4m3"):
    """Bit-exact when pre32 is None; otherwise one-step flips allowed near rounding boundaries."""
    g = codes(got) if not isinstance(got, np.ndarray) else got.astype(np.int64)
    w = np.asarray(want_codes, np.int64)
    diff = g != w
    if pre32 is None:
        assert not diff.any(), f"{what}: {int(diff.sum())} codes differ (bit-exact expected)"
        return 0
    n = int(diff.sum())
    if n == 0:
        return 0
    steps = np.abs(e4m3_step(g[diff]) - e4m3_step(w[diff]))
    # +0 and -0 are one "step" apart in value terms
    assert steps.max() <= 1 or np.all((g[diff] & 0x7F) + (w[diff] & 0x7F) <= 1), \
        f"{what}: codes differ by {int(steps.max())} steps"
    dist = nx.e4m3_midpoint_distance(np.asarray(pre32, np.float32)[diff], scale)
    assert np.all(dist <= near), (f"{what}: {int((dist > near).sum())} flips away from a "
                                  f"rounding boundary (max rel distance {dist.max():.2e})")
    assert n <= max(1, max_frac * g.size), f"{what}: {n} of {g.size} codes flipped"
    return n


def to_dev(t, device="cuda"):
    return t.to(device).contiguous()
