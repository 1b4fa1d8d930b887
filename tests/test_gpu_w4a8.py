"""The 8-bit-activation (W4A8) layer on the GPU vs the oracle's MXFP8 mode.

(1) moe_quant_mxfp8 gives the oracle's MXFP8 codes and scales bit for bit on
bf16 rows (random values over many binades, zero blocks, blocks whose maximum
rounds into the saturation range, subnormal results). (2) moe_forward_w4a8 on
small shapes and on the T = 4096 prefill workload: routing as in the bf16
tests, y against oracle.moe with act_mxfp8=True (x and h quantised to MXFP8
before the routed GEMMs) within relative L2 5e-3 and max |err| 2e-2 * rms.
(3) The quantisation is really applied: the W4A8 output differs from the
bf16 oracle by the size MXFP8 errors have.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle_par
import workloads as wl
from oracle import moe as omoe
from oracle import mxfp8

pytestmark = pytest.mark.gpu

REL_L2 = 5e-3
MAX_ABS = 2e-2


@pytest.fixture(scope="module")
def mx():
    import mxfp4_expert_gb300 as mx
    return mx


def test_quant_mxfp8_bit_exact(mx):
    g = torch.Generator().manual_seed(4)
    rows, K = 64, 512
    x = torch.randn((rows, K), generator=g) * torch.exp2(torch.randint(-20, 20, (rows, 1), generator=g).float())
    x[3, 32:64] = 0.0                                   # an all-zero block
    x[5, 0] = 480.0 * 2.0 ** -3                         # maximum in the saturation range after scaling
    x[6, :32] = torch.linspace(-1, 1, 32) * 2.0 ** -120  # tiny block: subnormal E4M3 results
    xb = x.to(torch.bfloat16)
    codes, scales = mx.moe_quant_mxfp8(xb.cuda())
    torch.cuda.synchronize()
    rc, rs = mxfp8.quantize(omoe.as_f64(xb))
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


def _check_w4a8(mx, w, set_idx, tokens=None):
    from mxfp4_expert_gb300 import synthetic
    layer = synthetic.build_layer(w, set_idx)
    x, bias = synthetic.inputs(w, set_idx)
    T, E, k = w.T, w.E, w.k
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = mx.moe_forward_w4a8(layer, x, bias, logits_out=logits, idx_out=idx, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    tokens = list(range(T)) if tokens is None else list(tokens)
    gi = idx.cpu().numpy()[tokens]
    b = None if bias is None else bias.cpu().numpy()
    if b is not None and b.ndim == 2:
        b = b[tokens]
    ri, _, _ = omoe.route_topk(logits.cpu().numpy()[tokens], k, b)
    assert np.array_equal(gi, ri)
    xs = x[tokens].cpu()
    router = wl.gen_router(w, set_idx, "cuda").cpu()
    shared = tuple(t.cpu() for t in wl.gen_shared(w, set_idx, "cuda"))
    ref = oracle_par.reference_layer(w, set_idx, xs, router, shared, b, gi, act_mxfp8=True)["y"]
    plain = oracle_par.reference_layer(w, set_idx, xs, router, shared, b, gi)["y"]
    yg = y.float().cpu().numpy().astype(np.float64)[tokens]
    rel = np.linalg.norm(yg - ref) / np.linalg.norm(ref)
    rms = np.sqrt(np.mean(ref ** 2))
    err = np.abs(yg - ref)
    within = err <= MAX_ABS * rms
    rounded = yg == oracle_par.bf16_rne(ref)
    assert rel <= REL_L2, rel
    assert np.all(within | rounded), (int((~(within | rounded)).sum()), float(err.max() / rms))
    q_err = np.linalg.norm(plain - ref) / np.linalg.norm(ref)
    assert q_err > 3 * rel, (q_err, rel)
    print(f"{w.name} w4a8: rel-L2 {rel:.2e} vs MXFP8 oracle, max|err|/rms {err.max() / rms:.2e}; "
          f"MXFP8 vs bf16 oracle {q_err:.2e}")


@pytest.mark.parametrize("name,T,d,I,E,k", [
    ("w4a8_tiny", 1, 512, 128, 32, 4),
    ("w4a8_small", 40, 512, 128, 32, 4),
    ("w4a8_ragged", 33, 512, 96, 24, 5),
    ("w4a8_many_rows", 300, 256, 64, 4, 2),
])
def test_w4a8_small(mx, name, T, d, I, E, k):
    w = wl.Workload(name, T=T, d=d, I=I, E=E, k=k, sets=1, routing="natural", seed=7)
    _check_w4a8(mx, w, 0)


def test_w4a8_ling_t64(mx):
    w = dataclasses.replace(wl.WORKLOADS["zipf_t64"], name="w4a8_zipf_t64")
    _check_w4a8(mx, w, 0)


@pytest.mark.slow
def test_w4a8_prefill_t4096(mx):
    w = wl.get("prefill_t4096")
    _check_w4a8(mx, w, 0, tokens=range(0, 4096, 16))
