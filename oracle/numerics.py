"""Number formats of the oracle: fp32, bf16 and FP8 E4M3 rounding, and per-tensor scaling.

Test infrastructure, never product code (see ``oracle/__init__.py``).

Everything here is written from the definition of the format, in float64 numpy, so that every
intermediate is exact: a value that is representable in fp32 is exact in float64, and scaling
by a power of two is exact.

The pages (TransformerEngine JAX Activation page, Description; LayerNorm Dense page,
Description) say only that tensors are quantized to FP8 before a GEMM and dequantized after
it.  The format and the recipe are left open; this oracle fixes them as: E4M3 ("fn" variant:
no infinities, one NaN pattern per sign), round to nearest even, saturating to +-448, with one
fp32 scale per tensor, scale = 448 / amax.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def to_f32(x) -> np.ndarray:
    """Round to the nearest fp32 (ties to even), returned as float64 holding fp32 values."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def _pow2_floor_exponent(a: np.ndarray) -> np.ndarray:
    """floor(log2(a)) for finite a > 0, exactly (frexp gives a = m * 2**e with m in [0.5, 1))."""
    _, e = np.frexp(a)
    return e.astype(np.int64) - 1


def bf16_round(x) -> np.ndarray:
    """fp32 -> bf16, round to nearest even (8 significant bits, fp32's exponent range).

    The grid spacing at |x| in [2**e, 2**(e+1)) is 2**(e-7); below 2**-126 the subnormal
    spacing 2**-133 applies.  A result past the largest finite bf16 becomes infinity, as IEEE
    round-to-nearest requires.  NaN stays NaN.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, dtype=np.float64, copy=True)
    fin = np.isfinite(x) & (x != 0)
    a = np.abs(x[fin])
    e = _pow2_floor_exponent(a)
    spacing = np.ldexp(1.0, np.maximum(e - 7, -133))
    r = np.rint(a / spacing) * spacing
    r = np.where(r > BF16_MAX, np.inf, r)
    out[fin] = np.copysign(r, x[fin])
    return out


def e4m3_decode(codes) -> np.ndarray:
    """E4M3 byte -> value.  Bits: sign s, exponent E (4 bits, bias 7), mantissa m (3 bits).

    E == 0: (-1)**s * m/8 * 2**-6 (subnormal).  Otherwise (-1)**s * (1 + m/8) * 2**(E-7),
    except E == 15, m == 7, which is NaN.
    """
    c = np.asarray(codes, dtype=np.int64) & 0xFF
    s = np.where(c & 0x80, -1.0, 1.0)
    E = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    val = np.where(E == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.ldexp(1.0, E - 7))
    val = np.where((E == 15) & (m == 7), np.nan, val)
    return s * val


def e4m3_encode(v) -> np.ndarray:
    """fp32 value -> E4M3 byte: round to nearest even, saturate to +-448 (satfinite).

    * NaN -> 0x7F with the sign bit of the input.
    * |v| >= 448 (including infinity) -> 448 with the input's sign.  Every value in
      (448, 464) is nearer to 448 than to the next grid point 480, 464 itself ties to the even
      mantissa of 448, and anything larger would round to 480, which is not finite in E4M3:
      saturation maps all of them to 448.
    * |v| < 2**-6: subnormal, code = round_half_even(|v| * 2**9); a result of 8 is the
      smallest normal (code 0x08), which the same formula produces.
    * otherwise, with e = floor(log2|v|): mantissa q = round_half_even((|v|/2**e - 1) * 8);
      q == 8 carries into the exponent.  code = (e + 7) << 3 | q.
    -0 keeps its sign (0x80).
    """
    v = np.asarray(v, dtype=np.float64)
    flat = v.reshape(-1)
    out = np.zeros(flat.shape, dtype=np.int64)
    sign = np.signbit(flat).astype(np.int64) << 7
    a = np.abs(flat)
    nan = np.isnan(flat)
    sat = ~nan & (a >= E4M3_MAX)
    sub = ~nan & (a < 2.0 ** -6)
    nrm = ~nan & ~sat & ~sub
    out[nan] = 0x7F
    out[sat] = 0x7E
    out[sub] = np.rint(a[sub] * 2.0 ** 9).astype(np.int64)
    an = a[nrm]
    e = _pow2_floor_exponent(an)
    q = np.rint((an / np.ldexp(1.0, e) - 1.0) * 8.0).astype(np.int64)
    carry = q == 8
    e = e + carry
    q = np.where(carry, 0, q)
    out[nrm] = ((e + 7) << 3) | q
    return (out | sign).astype(np.uint8).reshape(v.shape)


def compute_scale(amax) -> tuple[np.float32, np.float32]:
    """Per-tensor scale from an amax, in fp32 arithmetic: scale = 448 / amax.

    amax == 0 or not finite -> scale 1 (nothing to scale).  A quotient that overflows fp32
    (tiny amax) -> the largest finite fp32.  Returns (scale, scale_inv = 1 / scale).
    """
    amax = np.float32(amax)
    if not np.isfinite(amax) or amax == 0:
        s = np.float32(1.0)
    else:
        with np.errstate(over="ignore"):
            s = np.float32(E4M3_MAX) / amax
        if not np.isfinite(s):
            s = np.float32(np.finfo(np.float32).max)
    with np.errstate(over="ignore", divide="ignore"):
        s_inv = np.float32(1.0) / s
    return s, s_inv


def amax_of(v32) -> np.float32:
    """max |v| over a tensor of fp32 values (NaN ignored); 0 for an empty tensor."""
    a = np.abs(np.asarray(v32, dtype=np.float64))
    a = a[~np.isnan(a)]
    return np.float32(a.max()) if a.size else np.float32(0.0)


def quantize(v32, scale) -> np.ndarray:
    """E4M3 codes of fp32 values v with a given fp32 scale: encode(fp32(v * scale)).

    The product is taken in fp32, as the kernel takes it, so both sides decide each code from
    the same fp32 number.
    """
    prod = np.asarray(v32, dtype=np.float32) * np.float32(scale)
    return e4m3_encode(prod.astype(np.float64))


def dequantize(codes, scale_inv) -> np.ndarray:
    """fp32(decode(code) * scale_inv), as float64."""
    return to_f32(e4m3_decode(codes).astype(np.float32) * np.float32(scale_inv))
