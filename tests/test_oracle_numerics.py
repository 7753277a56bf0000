"""Pins for the oracle's number formats (oracle/numerics.py), against things other than itself.

* E4M3 encoding: brute-force nearest-of-all-finite-codes search (ties to the even code) over a
  stratified-exhaustive set of fp32 bit patterns; torch's float8_e4m3fn conversion (a library
  routine) where it is defined the same way (|v| <= 448); and the format's fixed points from the
  OCP 8-bit floating point specification (tests/golden/e4m3_points.txt).
* bf16 rounding: torch's fp32 -> bfloat16 conversion over the same stratified set.
* Scaling: closed-form cases of scale = 448 / amax.
"""

import os

import numpy as np
import pytest
import torch

from oracle import numerics as nx

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def stratified_f32_bits():
    """Every sign/exponent/top-7-mantissa-bit pattern (2**16) combined with low 16 mantissa
    bits chosen to sit on, just below and just above every rounding boundary of a format with
    up to 7 explicit mantissa bits (bf16), plus a few arbitrary ones.  For E4M3 (3 mantissa
    bits) the boundary bits lie in the top 16 bits, which are enumerated exhaustively."""
    hi = np.arange(1 << 16, dtype=np.uint64) << np.uint64(16)
    lo = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x1234, 0xC3A5],
                  dtype=np.uint64)
    bits = (hi[:, None] | lo[None, :]).reshape(-1).astype(np.uint32)
    return bits


def f32_from_bits(bits):
    with np.errstate(invalid="ignore"):
        return bits.view(np.float32).astype(np.float64)


def brute_force_e4m3(v):
    """Nearest finite E4M3 magnitude by exhaustive search; ties -> even code; sign copied."""
    codes = np.arange(0, 0x7F)  # all non-negative finite codes 0x00..0x7E
    mags = nx.e4m3_decode(codes)
    out = np.empty(v.shape, dtype=np.int64)
    a = np.abs(v)
    for s in range(0, len(v), 1 << 16):
        aa = a[s:s + (1 << 16)]
        d = np.abs(aa[:, None] - mags[None, :])
        best = d.min(axis=1, keepdims=True)
        cand = d == best
        # among equally near codes take the one whose mantissa LSB is 0
        even = cand & ((codes[None, :] & 1) == 0)
        pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
        out[s:s + len(aa)] = codes[pick]
    # above twice the largest finite magnitude every code lies below |v|, so the nearest is
    # the largest one (fp64 distances would no longer resolve 1-unit differences up there)
    out[a > 2 * mags.max()] = 0x7E
    sign = np.signbit(v).astype(np.int64) << 7
    return (out | sign).astype(np.uint8)


def test_e4m3_encode_matches_brute_force():
    bits = stratified_f32_bits()
    v = f32_from_bits(bits)
    keep = ~np.isnan(v)
    v = v[keep]
    got = nx.e4m3_encode(v)
    want = brute_force_e4m3(np.where(np.isinf(v), np.sign(v) * 1e30, v))
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (v[bad[:5]], got[bad[:5]], want[bad[:5]])


def test_e4m3_encode_matches_torch_in_range():
    bits = stratified_f32_bits()
    v = f32_from_bits(bits)
    keep = np.isfinite(v) & (np.abs(v) <= 448.0)
    v = v[keep]
    t = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = nx.e4m3_encode(v)
    assert np.array_equal(got, t)


def test_e4m3_nan_and_saturation():
    assert nx.e4m3_encode(np.array([np.nan]))[0] == 0x7F
    assert nx.e4m3_encode(np.array([-np.nan]))[0] == 0xFF
    for v, c in [(np.inf, 0x7E), (-np.inf, 0xFE), (1e38, 0x7E), (464.0, 0x7E), (449.0, 0x7E),
                 (-500.0, 0xFE)]:
        assert nx.e4m3_encode(np.array([v]))[0] == c, v


def test_e4m3_golden_points():
    """Fixed points of the E4M3 format (OCP OFP8 specification, E4M3 encoding table)."""
    rows = []
    with open(os.path.join(GOLDEN, "e4m3_points.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                val, code = line.split()
                rows.append((float.fromhex(val) if "p" in val else float(val), int(code, 16)))
    for val, code in rows:
        assert nx.e4m3_encode(np.array([val]))[0] == code, (val, hex(code))
        if abs(val) <= 448 and not np.isnan(val):
            # every listed in-range point is exactly representable or a documented tie
            dec = nx.e4m3_decode(np.array([code]))[0]
            assert abs(dec - val) <= abs(val) / 16 + 2.0 ** -10


def test_e4m3_decode_all_codes_roundtrip():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    vals = nx.e4m3_decode(codes)
    assert np.array_equal(nx.e4m3_encode(vals), codes.astype(np.uint8))
    t = torch.from_numpy(codes.astype(np.uint8)).view(torch.float8_e4m3fn).to(torch.float64)
    assert np.array_equal(t.numpy(), vals)
    assert np.isnan(nx.e4m3_decode(np.array([0x7F, 0xFF]))).all()


def test_bf16_round_matches_torch():
    bits = stratified_f32_bits()
    v32 = bits.view(np.float32)
    want = torch.from_numpy(v32.copy()).to(torch.bfloat16).to(torch.float64).numpy()
    with np.errstate(invalid="ignore"):
        got = nx.bf16_round(v32.astype(np.float64))
    both_nan = np.isnan(got) & np.isnan(want)
    assert np.array_equal(got[~both_nan], want[~both_nan])
    assert np.array_equal(np.isnan(got), np.isnan(want))


def test_to_f32_is_round_to_nearest():
    # 1 + 2**-24 is a tie between 1 and 1 + 2**-23: even mantissa (1) wins
    assert nx.to_f32(1.0 + 2.0 ** -24) == 1.0
    assert nx.to_f32(1.0 + 3 * 2.0 ** -24) == 1.0 + 2.0 ** -22


def test_compute_scale_cases():
    s, si = nx.compute_scale(0.0)
    assert s == 1.0 and si == 1.0
    s, si = nx.compute_scale(np.inf)
    assert s == 1.0
    s, si = nx.compute_scale(448.0)
    assert s == 1.0 and si == 1.0
    s, si = nx.compute_scale(1e-45)  # 448 / denormal overflows fp32
    assert s == np.finfo(np.float32).max
    s, si = nx.compute_scale(3.5)
    assert s == np.float32(128.0) and si == np.float32(1.0 / 128.0)


def test_amax_maps_to_max_code():
    """With scale = 448 / amax the element of largest magnitude always encodes as +-448."""
    rng = np.random.default_rng(1)
    amaxes = np.float32(np.exp(rng.uniform(-20, 20, size=2000)))
    for a in amaxes:
        s, _ = nx.compute_scale(a)
        assert nx.quantize(np.array([a, -a], np.float32), s).tolist() == [0x7E, 0xFE]


def test_quantize_dequantize_error_bound():
    """|dequant(quant(v)) - v| <= half an E4M3 step (relative 2**-4) for in-range normals."""
    rng = np.random.default_rng(2)
    v = rng.normal(size=100000).astype(np.float32)
    s, si = nx.compute_scale(nx.amax_of(v))
    back = nx.dequantize(nx.quantize(v, s), si)
    big = np.abs(v) * s >= 2.0 ** -6
    rel = np.abs(back[big] - v[big]) / np.abs(v[big])
    assert rel.max() <= 2.0 ** -4 * (1 + 1e-6)
