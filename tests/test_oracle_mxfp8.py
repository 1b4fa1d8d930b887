"""Pins for the MXFP8 (E4M3) activation mode of the oracle against torch's
float8_e4m3fn conversions (library routines)."""
import numpy as np
import torch

from oracle import mxfp8


def test_e4m3_decode_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = mxfp8.e4m3_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_rounding_matches_torch_rne():
    rng = np.random.default_rng(0)
    vals = mxfp8.e4m3_decode(np.arange(0x7F))
    mids = (vals[1:] + vals[:-1]) / 2
    q = np.concatenate([rng.uniform(-440, 440, 50000), rng.uniform(-0.1, 0.1, 20000),
                        mids, -mids, np.nextafter(mids, 0), np.nextafter(mids, 1000)])
    q = q.astype(np.float32).astype(np.float64)          # torch converts from fp32
    ref = torch.from_numpy(q.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = mxfp8.round_to_e4m3(q)
    assert np.array_equal(got, ref)


def test_mxfp8_block_scale_property():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((8, 256)) * np.exp(rng.uniform(-10, 10, (8, 1)))
    codes, s = mxfp8.quantize(x)
    amax = np.abs(x).reshape(8, 8, 32).max(-1)
    r = amax / np.ldexp(1.0, s.astype(np.int64) - 127)
    assert np.all((r >= 256) & (r < 512))
    fq = mxfp8.fake_quantize(x)
    rel = np.linalg.norm(fq - x) / np.linalg.norm(x)
    assert 0.005 < rel < 0.05          # E4M3 keeps 3 mantissa bits
