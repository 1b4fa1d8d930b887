"""FP8 LM-head GEMV in fp64 — TEST INFRASTRUCTURE.

Only tests, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline legs may use it.

Page "3 ways to speed up MoE inference on NVIDIA DGX Spark", §2 and §4: the
LM head projects the 2,560-wide hidden state onto 157,184 vocabulary logits;
the checkpoint keeps it in BF16, and quantising it online to FP8 halves the
bytes every decode step reads. The pages do not define the FP8 recipe; the
reading here is the usual per-output-channel one:

  * element: FP8 E4M3 (OCP: bias 7, 3 mantissa bits, largest finite 448);
  * scale: one fp32 number per output row v, s_v = fp32(amax_v / 448)
    (IEEE division in fp32, round to nearest even); a row of zeros gets s_v = 1;
  * code: E4M3 round-to-nearest-even of the fp32 quotient fp32(w / s_v),
    saturating at +-448;
  * logits[t, v] = s_v * sum_j x[t, j] * e4m3(code[v, j]), activations bf16
    (exact), everything after the quantisation exact in fp64.

Pins (tests/test_oracle_lmhead.py): codes against torch's float8_e4m3fn
conversion (a library routine) of the same fp32 quotients; the dequantised
row maximum is within one E4M3 step of amax; the GEMV against torch's float64
matmul on the dequantised weights; planted mistakes (scale not applied, scale
applied twice, transposed weights).
"""
from __future__ import annotations

import numpy as np

from . import mxfp8

E4M3_MAX = np.float32(448.0)


def quantize_rows(w) -> tuple[np.ndarray, np.ndarray]:
    """bf16-valued weights [V, d] -> (E4M3 codes uint8 [V, d], fp32 scales [V])."""
    w32 = np.asarray(w, dtype=np.float32)
    amax = np.max(np.abs(w32), axis=1).astype(np.float32)
    s = (amax / E4M3_MAX).astype(np.float32)               # fp32 division, RNE
    s = np.where(amax == 0, np.float32(1.0), s).astype(np.float32)
    q = (w32 / s[:, None]).astype(np.float32)              # fp32 division, RNE
    codes = mxfp8.round_to_e4m3(q.astype(np.float64))
    return codes, s


def dequantize_rows(codes, scales) -> np.ndarray:
    """Exact fp64 values of the quantised rows: e4m3(code) * s_v."""
    return mxfp8.e4m3_decode(codes) * np.asarray(scales, dtype=np.float64)[:, None]


def logits(x, codes, scales) -> np.ndarray:
    """fp64 logits [T, V] of activations x [T, d] against the FP8 head."""
    x64 = np.asarray(x, dtype=np.float64)
    return (x64 @ mxfp8.e4m3_decode(codes).T) * np.asarray(scales, dtype=np.float64)[None, :]
