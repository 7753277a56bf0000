"""Comparison rules between the CUDA path and the oracle.

* GEMM outputs (contraction K): max |gpu - ref| <= 2e-2 * sqrt(K) * rms(A) * rms(B), i.e. a
  2e-2 fraction of the output's expected magnitude; when the output is stored in bf16 on both
  sides, plus one bf16 ulp of the value (2**-8 * |ref|), since the two roundings may pick
  adjacent bf16 numbers.
* Elementwise bf16 outputs: |gpu - ref| <= 2e-2 * |ref| + 1e-3 * rms(ref).
* fp32 reductions (mu, rsigma, dbias, dgamma, dbeta): |gpu - ref| <= 1e-4 * max(|ref|, rms(ref)).
* E4M3 codes from identical fp32 inputs: bit-exact.  Codes of values the GPU computed itself
  (through a norm or a GEMM epilogue): equal, except at most one step apart on at most 0.1% of
  elements, and only where the oracle's pre-cast value lies within the test's fp32 error bound
  of a rounding boundary, so that fp32 evaluation-order differences can explain the flip.
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


def assert_gemm_close(got, ref, K, rms_a, rms_b, what="gemm", stored=None):
    """``stored`` = "bf16" when both sides rounded the result to bf16: they may then land on
    adjacent bf16 numbers, so one bf16 ulp of the stored value (2**-8 relative) is added."""
    if stored is None:
        stored = "bf16" if isinstance(got, torch.Tensor) and got.dtype == torch.bfloat16 else "f32"
    got, ref = np64(got), np.asarray(ref, np.float64)
    tol = 2e-2 * math.sqrt(K) * rms_a * rms_b
    if stored == "bf16":
        tol = tol + 2.0 ** -8 * np.abs(ref)
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    ratio = err / tol
    worst = float(ratio.max()) if err.size else 0.0
    assert worst <= 1.0, (f"{what}: max err/tol {worst:.3f} (max err {float(err.max()):.3e}, "
                          f"K={K})")
    return worst


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
    """Signed position of each code on the ordered E4M3 grid (so a one-step flip differs by 1).
    +0 and -0 share position 0."""
    c = np.asarray(c, np.int64)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


_GRID = np.unique(np.abs(nx.e4m3_decode(np.arange(0, 0x7F))))
_MIDS = (_GRID[:-1] + _GRID[1:]) / 2.0


def boundary_distance(v32, scale) -> np.ndarray:
    """|fp32(v * scale)| to the nearest E4M3 rounding boundary (a midpoint between adjacent
    finite E4M3 values), in the scaled domain."""
    y = np.abs(np.asarray(v32, dtype=np.float32) * np.float32(scale)).astype(np.float64)
    y = np.minimum(y, _GRID[-1])
    idx = np.clip(np.searchsorted(_MIDS, y), 1, len(_MIDS) - 1)
    return np.minimum(np.abs(y - _MIDS[idx - 1]), np.abs(y - _MIDS[idx]))


def assert_e4m3_codes(got, want_codes, pre32=None, scale=None, rel=1e-5, abs_tol=0.0,
                      max_frac=1e-3, what="e4m3"):
    """Bit-exact when ``pre32`` is None (identical fp32 inputs on both sides).

    Otherwise the GPU computed the pre-cast values itself, in fp32 and in its own order, so a
    code may sit one step away from the oracle's where the oracle's value v lies within
    ``rel * |v| + abs_tol`` of a rounding boundary (that bound is the test's estimate of the
    GPU's fp32 error on v), on at most ``max_frac`` of the elements.  +0 and -0 compare equal.
    """
    g = codes(got) if not isinstance(got, np.ndarray) else got.astype(np.int64)
    w = np.asarray(want_codes, np.int64)
    diff = e4m3_step(g) != e4m3_step(w)
    if pre32 is None:
        assert not diff.any(), f"{what}: {int(diff.sum())} codes differ (bit-exact expected)"
        return 0
    n = int(diff.sum())
    if n == 0:
        return 0
    steps = np.abs(e4m3_step(g[diff]) - e4m3_step(w[diff]))
    assert steps.max() <= 1, f"{what}: codes differ by up to {int(steps.max())} steps"
    v = np.asarray(pre32, np.float64)[diff]
    dist = boundary_distance(v, scale)
    if np.ndim(abs_tol):  # a window per element
        abs_tol = np.broadcast_to(np.asarray(abs_tol, np.float64), np.shape(pre32))[diff]
    allowed = (rel * np.abs(v) + abs_tol) * float(scale)
    far = dist > allowed
    assert not far.any(), (f"{what}: {int(far.sum())} of {n} flips farther from a rounding "
                           f"boundary than the fp32 error bound allows "
                           f"(worst {float((dist / np.maximum(allowed, 1e-300)).max()):.2f}x)")
    assert n <= max(1, max_frac * g.size), f"{what}: {n} of {g.size} codes flipped"
    return n


_DECODE = nx.e4m3_decode(np.arange(256))


def decode(c) -> np.ndarray:
    """nx.e4m3_decode by table lookup (the table is the oracle's decode of all 256 codes), for
    the large code tensors of the full-size tests."""
    return _DECODE[np.asarray(c, np.int64) & 0xFF]


def quantize_fast(v, scale) -> np.ndarray:
    """nx.quantize for large arrays of finite values, through torch's float8_e4m3fn conversion
    on the CPU: fp32(v * scale), clamped to +-448 (the recipe's saturation), then rounded to
    nearest even.  tests/test_oracle_numerics.py pins that conversion to the oracle's encoder
    for every |v| <= 448."""
    t = torch.from_numpy(np.ascontiguousarray(np.asarray(v, np.float32)))
    t = (t * torch.tensor(np.float32(scale))).clamp(-448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().astype(np.int64)


def to_dev(t, device="cuda"):
    return t.to(device).contiguous()


# ---------------------------------------------------------------------- error windows ------
#
# A value the GPU computes in fp32 differs from the oracle's float64 value by at most a known
# bound w (its fp32 error window).  Where it is then rounded (to bf16, or to an E4M3 code), the
# two roundings can differ only if the interval [v - w, v + w] straddles a rounding midpoint,
# and then only by the jump between the two rounded ends.  A consumer that is linear in such
# values inherits the jumps through the absolute values of its coefficients.  These windows let
# the tests compare each step of a chain with the oracle's step at the pages' tight rules,
# adding exactly what the rounding of an fp32 intermediate can explain.

# |fp32 GEMM result - exact| <= ACC_REL * sum_k |a_k b_k| for the library's tensor-core GEMMs
# (bf16 and E4M3 operands, fp32 accumulation); tests/test_gpu_kernels.py measures it.
ACC_REL = 2.0 ** -18


def gemm_window(a, b, alpha=1.0):
    """fp32 accumulation window of alpha * (a @ b): ACC_REL * |alpha| * (|a| @ |b|)."""
    return ACC_REL * abs(float(alpha)) * (np.abs(np.asarray(a, np.float64)) @
                                          np.abs(np.asarray(b, np.float64)))


def bf16_jump(v64, w) -> np.ndarray:
    """How far the bf16 rounding of a value known to within +-w of v64 can move from
    bf16(v64): 0 where [v - w, v + w] rounds to one bf16 number."""
    v = np.asarray(v64, np.float64)
    lo, hi, mid = nx.bf16_round(v - w), nx.bf16_round(v + w), nx.bf16_round(v)
    return np.maximum(np.abs(hi - mid), np.abs(mid - lo))


def assert_in_window(got, ref64, w, what, stored="f32", rel=1e-4, max_frac=None):
    """``got`` against the float64 reference ``ref64`` known to within +-w (array or scalar).

    stored="bf16": got must be a bf16 rounding of a value in [ref - w, ref + w] (rounding is
    monotonic, so bf16(ref - w) <= got <= bf16(ref + w)); ``max_frac`` bounds the fraction of
    elements that differ from bf16(ref) at all.
    stored="f32" (an fp32 reduction): |got - ref| <= rel * max(|ref|, rms(ref)) + w, the 1e-4
    reduction rule plus the window its inputs carry.
    """
    got, ref = np64(got), np.asarray(ref64, np.float64)
    w = np.broadcast_to(np.asarray(w, np.float64), ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    if stored == "bf16":
        lo, hi = nx.bf16_round(ref - w), nx.bf16_round(ref + w)
        bad = (got < lo) | (got > hi)
        assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outside the window; first "
                               f"got {got[bad][:3]} ref {ref[bad][:3]} w {w[bad][:3]}")
        if max_frac is not None:
            moved = got != nx.bf16_round(ref)
            assert moved.mean() <= max_frac, f"{what}: {int(moved.sum())} of {moved.size} moved"
        return
    scale = np.maximum(np.abs(ref), rms(ref))
    err = np.abs(got - ref)
    tol = rel * scale + w
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} out of tolerance; worst "
                           f"{float((err / tol).max()):.3f}x")


# ---------------------------------------------------------------------- guard bands --------

GUARD_BYTE = 0xA5


class Guarded:
    """An output tensor with guard bands on both sides: ``t`` is a contiguous view into a larger
    byte buffer whose first and last ``rows`` rows' worth of bytes (at least 4 KiB) hold
    GUARD_BYTE.  ``check()`` asserts that no byte of either band changed, so that a store past
    a tile edge of a ragged shape into neighbouring memory fails the test."""

    def __init__(self, shape, dtype, device="cuda", rows=256):
        esz = torch.tensor([], dtype=dtype).element_size()
        n = 1
        for d in shape:
            n *= int(d)
        row = int(shape[-1]) * esz if len(shape) else esz
        g = max(4096, rows * row)
        self.g = (g + 255) // 256 * 256
        self.nbytes = n * esz
        self.raw = torch.full((self.nbytes + 2 * self.g,), GUARD_BYTE, dtype=torch.uint8,
                              device=device)
        self.t = self.raw[self.g:self.g + self.nbytes].view(dtype).view(*shape)

    def check(self, what="output"):
        torch.cuda.synchronize()
        lo = self.raw[:self.g]
        hi = self.raw[self.g + self.nbytes:]
        nlo = int((lo != GUARD_BYTE).sum().item())
        nhi = int((hi != GUARD_BYTE).sum().item())
        assert nlo == 0 and nhi == 0, (f"{what}: {nlo} bytes before and {nhi} bytes after the "
                                       f"tensor were overwritten")
