"""MXFP8 (E4M3 elements, E8M0 scale per 32) activation quantisation — TEST INFRASTRUCTURE.

Only tests, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline legs may use it.

The pages' baseline MoE configuration is W4A8 (page "3 ways to speed up MoE
inference on NVIDIA DGX Spark", §2: "W4A8 configuration"), i.e. 8-bit
activations against 4-bit weights; they do not define the 8-bit format. This
module takes the OCP MX v1.0 MXFP8 E4M3 format: 1 sign, 4 exponent bits (bias
7), 3 mantissa bits; largest finite 448; S.1111.111 is NaN; exponent field 0
is subnormal (step 2^-9). Scale rule as for MXFP4 with emax_elem = 8:
X = 2^(floor(log2 amax) - 8); elements v/X rounded to nearest E4M3, ties to
even, saturating at +-448.

This is the oracle's "MXFP8 activations" mode: the W4A8 prefill path is
judged against it, the bf16 path against the plain oracle.

Pins: decoding of all 256 codes against torch's float8_e4m3fn conversion;
rounding of random values and every midpoint against torch's float8_e4m3fn
round-to-nearest-even conversion (a library routine) in the range where no
saturation applies.
"""
from __future__ import annotations

import numpy as np

E4M3_EMAX = 8
E4M3_MAX = 448.0
BLOCK = 32


def e4m3_decode(codes) -> np.ndarray:
    """E4M3 byte -> fp64 value (0x7F / 0xFF -> NaN)."""
    c = np.asarray(codes, dtype=np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return s * mag


# all finite non-negative E4M3 magnitudes, ascending, with their codes
_POS_CODES = np.array([c for c in range(0x7F)], dtype=np.int64)     # 0x00..0x7E
_POS_VALUES = e4m3_decode(_POS_CODES)


def round_to_e4m3(q: np.ndarray) -> np.ndarray:
    """Nearest E4M3 code for fp64 q (ties to even code, saturate at 448, keep sign)."""
    q = np.asarray(q, dtype=np.float64)
    a = np.minimum(np.abs(q), E4M3_MAX)
    pos = np.searchsorted(_POS_VALUES, a)              # first value >= a
    pos = np.clip(pos, 1, len(_POS_VALUES) - 1)
    lo, hi = _POS_VALUES[pos - 1], _POS_VALUES[pos]
    dlo, dhi = a - lo, hi - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & ((_POS_CODES[pos] & 1) == 0))
    code = np.where(pick_hi, _POS_CODES[pos], _POS_CODES[pos - 1])
    code = np.where(a == 0.0, 0, code)
    return (code | (np.signbit(q).astype(np.int64) << 7)).astype(np.uint8)


def quantize(x: np.ndarray):
    """MXFP8 quantisation of x [..., K] row-wise: (codes [..., K] uint8, scales [..., K/32] uint8)."""
    v = np.asarray(x, dtype=np.float64)
    K = v.shape[-1]
    v = v.reshape(*v.shape[:-1], K // BLOCK, BLOCK)
    amax = np.max(np.abs(v), axis=-1)
    _, e = np.frexp(amax)
    s = np.clip(e.astype(np.int64) - 1 - E4M3_EMAX + 127, 0, 254)
    s = np.where(amax == 0.0, 0, s)
    X = np.ldexp(1.0, s - 127)
    codes = round_to_e4m3(v / X[..., None]).reshape(*v.shape[:-2], K)
    return codes, s.astype(np.uint8)


def fake_quantize(x: np.ndarray) -> np.ndarray:
    """dequantize(quantize(x)) in fp64."""
    codes, s = quantize(x)
    K = codes.shape[-1]
    return e4m3_decode(codes) * np.repeat(np.ldexp(1.0, s.astype(np.int64) - 127), BLOCK, axis=-1)
