"""Pins for the FP8 LM-head oracle against torch library routines and planted mistakes."""
import numpy as np
import torch

from oracle import lmhead, mxfp8


def _weights(V=96, d=256, seed=0):
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((V, d)) * np.exp(rng.uniform(-6, 2, (V, 1)))
    w[3] = 0.0                                         # a zero row
    w[5, 7] = 40.0 * np.abs(w[5]).max()                # one outlier
    return torch.from_numpy(w).to(torch.bfloat16).to(torch.float64).numpy()


def test_codes_match_torch_float8_conversion():
    w = _weights()
    codes, s = lmhead.quantize_rows(w)
    q = torch.from_numpy(w.astype(np.float32)) / torch.from_numpy(s)[:, None]   # fp32 division
    ref = q.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)
    assert s[3] == 1.0 and np.all(codes[3] & 0x7F == 0)


def test_row_maximum_is_kept():
    w = _weights(seed=1)
    codes, s = lmhead.quantize_rows(w)
    deq = lmhead.dequantize_rows(codes, s)
    amax = np.abs(w).max(1)
    got = np.abs(deq).max(1)
    ok = amax > 0
    assert np.all(np.abs(got[ok] - amax[ok]) <= amax[ok] / 16)   # one E4M3 step at the top binade
    rel = np.linalg.norm(deq - w) / np.linalg.norm(w)
    assert rel < 0.05


def test_logits_match_torch_matmul_on_dequantised_weights():
    w = _weights(seed=2)
    codes, s = lmhead.quantize_rows(w)
    x = torch.randn((3, w.shape[1]), generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    x64 = x.to(torch.float64)
    got = lmhead.logits(x64.numpy(), codes, s)
    ref = (x64 @ torch.from_numpy(lmhead.dequantize_rows(codes, s)).T).numpy()
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)
    # planted mistakes
    x64n = x64.numpy()
    no_scale = x64n @ mxfp8.e4m3_decode(codes).T
    twice = got * s[None, :]
    for bad in (no_scale, twice):
        assert np.linalg.norm(bad - got) > 1e-3 * np.linalg.norm(got)
