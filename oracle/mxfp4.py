"""MXFP4 arithmetic in fp64 — oracle for packing and dequantisation. TEST INFRASTRUCTURE.

Only tests, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline legs may use it.

The pages describe the experts of Ling-3.0-flash as stored in MXFP4 (page
"3 ways to speed up MoE inference on NVIDIA DGX Spark", §2 and §3) but never
define the format. The definition used here is the public OCP Microscaling
Formats (MX) Specification v1.0:

  * element: FP4 E2M1 — 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit,
    no inf/NaN. Magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}; exponent field 0 is
    subnormal (0 and 0.5).
  * scale: E8M0 — an unsigned 8-bit biased exponent, value 2^(s-127);
    s = 255 is NaN.
  * block: 32 consecutive elements along K share one scale.
  * quantisation (spec §6.3): X = 2^(floor(log2(amax)) - emax_elem) with
    emax_elem = 2 for E2M1, then every element is v/X rounded to the nearest
    E2M1 value, ties to even, saturating at +-6. amax = 0 gives s = 0.
    A block holding a non-finite value gets the NaN scale 255.

Canonical byte layout used by the oracle (and by the library's unpack call):
codes [N, K/2] uint8 with element 2j in the low nibble of byte j and element
2j+1 in the high nibble; scales [N, K/32] uint8.

Pins (tests/test_oracle_mxfp4.py): exhaustive 16 codes x 255 scales against
torch's float8_e8m0fnu conversion and the E2M1 value set; rounding against the
FPU's own round-to-nearest-even at the mantissa position; every midpoint +-1
ulp; the OCP binade property of the chosen scale; value idempotence; planted
mistakes.
"""
from __future__ import annotations

import numpy as np

# E2M1 magnitudes indexed by the low 3 code bits (e1 e0 m). The mantissa bit
# is code & 1, so "even" codes are 0, 2, 4, 6.
E2M1_MAGNITUDE = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)
E2M1_EMAX = 2          # largest normal exponent: 6 = 1.5 * 2^2
E8M0_BIAS = 127
E8M0_NAN = 255
BLOCK = 32


def e2m1_decode(codes) -> np.ndarray:
    """E2M1 code (0..15) -> value, fp64. Bit 3 is the sign."""
    c = np.asarray(codes, dtype=np.int64)
    mag = E2M1_MAGNITUDE[c & 7]
    return np.where(c & 8, -mag, mag)


def e8m0_decode(s) -> np.ndarray:
    """E8M0 scale byte -> 2^(s-127), fp64; 255 -> NaN."""
    s = np.asarray(s, dtype=np.int64)
    v = np.ldexp(1.0, s - E8M0_BIAS)
    return np.where(s == E8M0_NAN, np.nan, v)


def unpack_nibbles(codes_packed: np.ndarray) -> np.ndarray:
    """[..., K/2] bytes -> [..., K] codes; element 2j is the low nibble of byte j."""
    b = np.asarray(codes_packed, dtype=np.uint8)
    lo = b & 0x0F
    hi = b >> 4
    return np.stack([lo, hi], axis=-1).reshape(*b.shape[:-1], b.shape[-1] * 2)


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """[..., K] codes -> [..., K/2] bytes (inverse of unpack_nibbles)."""
    c = np.asarray(codes, dtype=np.uint8)
    c = c.reshape(*c.shape[:-1], c.shape[-1] // 2, 2)
    return (c[..., 0] | (c[..., 1] << 4)).astype(np.uint8)


def dequantize(codes_packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Exact fp64 values of MXFP4 data: value = e2m1(code) * 2^(s-127).

    codes_packed [..., K/2] uint8, scales [..., K/32] uint8 -> [..., K] fp64.
    """
    codes = unpack_nibbles(codes_packed)
    vals = e2m1_decode(codes)
    sc = np.repeat(e8m0_decode(scales), BLOCK, axis=-1)
    return vals * sc


def scale_exponent(amax: np.ndarray) -> np.ndarray:
    """OCP MX scale byte for blocks with absolute maximum amax (finite, >= 0).

    s = floor(log2(amax)) - emax_elem + 127, clamped to the E8M0 range
    [0, 254]; amax = 0 gives 0. floor(log2) is read exactly from frexp:
    amax = f * 2^e with f in [0.5, 1) means floor(log2(amax)) = e - 1.
    """
    a = np.asarray(amax, dtype=np.float64)
    _, e = np.frexp(a)
    s = (e.astype(np.int64) - 1) - E2M1_EMAX + E8M0_BIAS
    s = np.clip(s, 0, 254)
    return np.where(a == 0.0, 0, s).astype(np.int64)


def round_to_e2m1(q: np.ndarray) -> np.ndarray:
    """Nearest E2M1 code for fp64 values q: ties to the even mantissa, saturating.

    The sign bit of q is kept (so small negatives give code 8, i.e. -0).
    Written as the definition: among the two grid magnitudes around |q| the
    nearer wins, and on a tie the code with mantissa bit 0 wins. Magnitudes
    above 6 saturate to 6 (spec: conversion to E2M1 saturates).
    """
    q = np.asarray(q, dtype=np.float64)
    a = np.minimum(np.abs(q), 6.0)
    hi = np.clip(np.searchsorted(E2M1_MAGNITUDE, a), 1, 7)   # first magnitude >= a
    lo = hi - 1
    d_lo = a - E2M1_MAGNITUDE[lo]
    d_hi = E2M1_MAGNITUDE[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((hi & 1) == 0))
    mag = np.where(pick_hi, hi, lo)
    sign = np.signbit(q).astype(np.int64) << 3
    return (mag | sign).astype(np.uint8)


def quantize(w: np.ndarray):
    """MX quantisation of fp32 weights w [..., K] (K % 32 == 0), row-wise blocks.

    Returns (codes_packed [..., K/2] uint8, scales [..., K/32] uint8,
    nonfinite: bool). Steps, per 32-element block:
      1. amax = max |v| (exact).
      2. s = scale_exponent(amax); X = 2^(s-127).
      3. q = v / X, exact in fp64 (X is a power of two).
      4. code = round_to_e2m1(q).
    A block containing inf or NaN gets scale 255 and codes from its finite
    values treated as above; the returned flag reports it.
    """
    w = np.asarray(w, dtype=np.float32)
    K = w.shape[-1]
    assert K % BLOCK == 0, "K must be a multiple of 32"
    v = w.astype(np.float64).reshape(*w.shape[:-1], K // BLOCK, BLOCK)
    finite = np.isfinite(v)
    amax = np.max(np.where(finite, np.abs(v), 0.0), axis=-1)
    s = scale_exponent(amax)
    X = np.ldexp(1.0, s - E8M0_BIAS)
    q = np.where(finite, v, 0.0) / X[..., None]
    codes = round_to_e2m1(q)
    bad = ~finite.all(axis=-1)
    s = np.where(bad, E8M0_NAN, s)
    codes = codes.reshape(*w.shape[:-1], K)
    return pack_nibbles(codes), s.astype(np.uint8), bool(bad.any())


def fake_quantize(w: np.ndarray) -> np.ndarray:
    """dequantize(quantize(w)) — the fp64 values the layer actually multiplies by."""
    c, s, _ = quantize(w)
    return dequantize(c, s)
