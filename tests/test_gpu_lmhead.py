"""FP8 LM head on the GPU vs the oracle (oracle.lmhead).

(1) moe_lmhead_pack_fp8 gives the oracle's codes and scales bit for bit
(random bf16 rows over many binades, a zero row, a row with one outlier).
(2) moe_lmhead_fp8 at T = 1..8 against the oracle's fp64 logits on the same
codes: |err| <= 1e-5 * sum_j |x_j w_j| per logit (fp32 accumulation of exact
products), on a small head and on the Ling head (V = 157,184, d = 2,560)
sampled rows. (3) Deterministic: two calls give identical bits.
"""
import numpy as np
import pytest
import torch

from oracle import lmhead, mxfp8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    import mxfp4_expert_gb300 as mx
    return mx


def _head(V, d, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    w = (torch.randn((V, d), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    return w


def test_pack_bit_exact(mx):
    g = torch.Generator().manual_seed(1)
    V, d = 64, 256
    w = torch.randn((V, d), generator=g) * torch.exp2(torch.randint(-12, 6, (V, 1), generator=g).float())
    w[2] = 0.0
    w[9, 17] = 300.0
    wb = w.to(torch.bfloat16)
    codes, scales = mx.moe_lmhead_pack_fp8(wb.cuda())
    torch.cuda.synchronize()
    rc, rs = lmhead.quantize_rows(wb.to(torch.float64).numpy())
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


def _check(mx, V, d, T, rows=None, seed=0):
    w = _head(V, d, seed)
    codes, scales = mx.moe_lmhead_pack_fp8(w)
    x = torch.randn((T, d), generator=torch.Generator().manual_seed(seed + 1)).to(torch.bfloat16).cuda()
    y = mx.moe_lmhead_fp8(codes, scales, x)
    y2 = mx.moe_lmhead_fp8(codes, scales, x)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int32), y2.view(torch.int32))
    rows = np.arange(V) if rows is None else np.asarray(rows)
    c = codes[rows].cpu().numpy()
    s = scales[rows].cpu().numpy()
    x64 = x.cpu().to(torch.float64).numpy()
    ref = lmhead.logits(x64, c, s)
    bound = 1e-5 * (np.abs(x64) @ np.abs(lmhead.dequantize_rows(c, s)).T)
    err = np.abs(y.cpu().numpy()[:, rows] - ref)
    assert np.all(err <= bound + 1e-30), float((err / (bound + 1e-30)).max())
    return float((err / (bound + 1e-30)).max())


@pytest.mark.parametrize("T", [1, 2, 3, 4, 8])
def test_gemv_small(mx, T):
    _check(mx, 512, 256, T, seed=T)


@pytest.mark.parametrize("T", [1, 4])
def test_gemv_ling_head(mx, T):
    V, d = 157184, 2560
    rng = np.random.default_rng(T)
    rows = np.concatenate([np.arange(32), rng.choice(V, 480, replace=False), np.arange(V - 32, V)])
    _check(mx, V, d, T, rows=rows, seed=10 + T)


def test_rejects_bad_shapes(mx):
    w = _head(48, 64, 0)
    codes, scales = mx.moe_lmhead_pack_fp8(w)
    x = torch.zeros((9, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mx.MoeError):
        mx.moe_lmhead_fp8(codes, scales, x)   # T > 8
