"""moe_pack_mxfp4 / moe_unpack_mxfp4 on the GPU vs. the oracle's MX quantisation: bit-exact."""
import numpy as np
import pytest
import torch

import workloads as wl
from oracle import mxfp4

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    import mxfp4_expert_gb300 as mx
    return mx


def gpu_pack_unpack(mx, w, layout):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    packed, desc = mx.moe_pack_mxfp4(w.cuda().contiguous(), layout, dev_status=st)
    codes, scales = mx.moe_unpack_mxfp4(packed, desc)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy(), int(st.item()), packed, desc


def check_exact(mx, w, layout):
    codes, scales, st, _, _ = gpu_pack_unpack(mx, w, layout)
    wn = w.numpy() if w.dim() == 3 else w.numpy()[None]
    rc, rs, bad = mxfp4.quantize(wn)
    assert np.array_equal(scales, rs), "scale bytes differ"
    assert np.array_equal(codes, rc), "code bytes differ"
    return st, bad


@pytest.mark.parametrize("n_mat,N,K,layout", [
    (1, 16, 32, 1), (3, 48, 96, 1), (2, 32, 64, 2), (4, 256, 512, 2), (2, 512, 128, 1),
    (1, 16, 2560, 1), (5, 1536, 2560 // 8, 2)])
def test_pack_random_bit_exact(mx, n_mat, N, K, layout):
    g = torch.Generator().manual_seed(N * 7 + K)
    w = torch.randn((n_mat, N, K), generator=g) * 0.02
    # vary magnitudes per row so many scale bytes appear
    w = w * torch.exp2(torch.randint(-30, 30, (n_mat, N, 1), generator=g).float())
    st, _ = check_exact(mx, w, layout)
    assert st == 0


def test_pack_thresholds_signs_and_extremes(mx):
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    rows = []
    for scale in [1.0, 2.0 ** -20, 2.0 ** 40]:
        for m in mids:
            lo, hi = np.nextafter(np.float32(m), np.float32(0)), np.nextafter(np.float32(m), np.float32(8))
            r = np.zeros(32, dtype=np.float32)
            r[0] = 6.0
            r[1:4] = [m, lo, hi]
            r[4:7] = [-m, -lo, -hi]
            r[7] = -0.0
            r[8] = -1e-9
            r[9] = 7.5          # saturates to 6
            rows.append(r * np.float32(scale))
    rows.append(np.zeros(32, dtype=np.float32))                       # all-zero block -> s = 0
    rows.append(np.full(32, 1e-40, dtype=np.float32))                 # subnormal amax -> s = 0
    rows.append(np.full(32, -3e-39, dtype=np.float32))
    rows.append(np.linspace(-1e30, 1e30, 32, dtype=np.float32))
    while len(rows) % 16:
        rows.append(np.zeros(32, dtype=np.float32))
    w = torch.from_numpy(np.stack(rows))[None]
    st, _ = check_exact(mx, w, 1)
    assert st == 0


def test_pack_nonfinite_and_scale_range_flags(mx):
    w = torch.randn((1, 16, 64)) * 0.02
    w[0, 3, 40] = float("nan")
    w[0, 5, 1] = float("inf")
    codes, scales, st, _, _ = gpu_pack_unpack(mx, w, 1)
    assert st & mx.DEV_NONFINITE_INPUT
    assert scales[0, 3, 1] == 255 and scales[0, 5, 0] == 255 and scales[0, 3, 0] != 255
    rc, rs, bad = mxfp4.quantize(w.numpy())
    assert bad and np.array_equal(scales, rs) and np.array_equal(codes, rc)
    w2 = torch.randn((1, 16, 32)) * 0.02
    w2[0, 0, 0] = 3e37
    _, s2, st2, _, _ = gpu_pack_unpack(mx, w2, 1)
    assert st2 & mx.DEV_SCALE_RANGE and s2[0, 0, 0] > 248


def test_pack_ling_expert_sample(mx):
    w = wl.get("ling_t1")
    for e in (0, 137, 511):
        gu, dn = wl.gen_expert(w, 0, e, "cuda")
        c1, s1, st1, _, _ = gpu_pack_unpack(mx, gu[None], 2)
        c2, s2, st2, _, _ = gpu_pack_unpack(mx, dn[None], 1)
        rc1, rs1, _ = mxfp4.quantize(gu.cpu().numpy()[None])
        rc2, rs2, _ = mxfp4.quantize(dn.cpu().numpy()[None])
        assert st1 == 0 and st2 == 0
        assert np.array_equal(s1, rs1) and np.array_equal(c1, rc1)
        assert np.array_equal(s2, rs2) and np.array_equal(c2, rc2)


def test_pack_rejects_bad_arguments(mx):
    w = torch.randn((1, 20, 64), device="cuda")
    with pytest.raises(mx.MoeError):
        mx.moe_pack_mxfp4(w, 1)                        # N % 16 != 0
    w = torch.randn((1, 16, 64), device="cuda")
    small = torch.empty(10, dtype=torch.uint8, device="cuda")
    with pytest.raises(mx.MoeError):
        mx.moe_pack_mxfp4(w, 1, out=small)             # buffer too small


def packed_reference(codes, scales, layout):
    """The packed bytes as include/moe_mxfp4.h documents them, built from the
    oracle's canonical codes [n_mat][N][K/2] and scales [n_mat][N][K/32]:
    unit (tile r, block b) at (r*K/32 + b)*272; bytes [16i, 16i+16) = packed row
    i's canonical bytes of block b; byte 256 + 2g + h = scale of row g + 8h.
    GATEUP: packed row i of tile r is gate row 8r + i (i < 8) or up row
    I + 8r + i - 8."""
    n_mat, N, KH = codes.shape
    KB = KH // 16
    out = np.zeros(n_mat * N * KB * 272 // 16, dtype=np.uint8)
    o = 0
    for m in range(n_mat):
        for r in range(N // 16):
            for b in range(KB):
                unit = np.zeros(272, dtype=np.uint8)
                for i in range(16):
                    if layout == 2:
                        src = 8 * r + i if i < 8 else N // 2 + 8 * r + i - 8
                    else:
                        src = 16 * r + i
                    unit[16 * i:16 * i + 16] = codes[m, src, 16 * b:16 * b + 16]
                    g, h = (i, 0) if i < 8 else (i - 8, 1)
                    unit[256 + 2 * g + h] = scales[m, src, b]
                out[o:o + 272] = unit
                o += 272
    return out


@pytest.mark.parametrize("n_mat,N,K,layout", [(2, 32, 96, 1), (1, 48, 64, 2), (1, 64, 256, 2)])
def test_pack_bytes_match_documented_layout(mx, n_mat, N, K, layout):
    """The raw packed bytes (not their unpacking) against the header's layout
    formula applied to the oracle's quantisation."""
    g = torch.Generator().manual_seed(N + K + layout)
    w = torch.randn((n_mat, N, K), generator=g) * 0.02
    w = w * torch.exp2(torch.randint(-8, 8, (n_mat, N, 1), generator=g).float())
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    packed, _ = mx.moe_pack_mxfp4(w.cuda().contiguous(), layout, dev_status=st)
    torch.cuda.synchronize()
    rc, rs, _ = mxfp4.quantize(w.numpy())
    ref = packed_reference(rc, rs, layout)
    got = packed.cpu().numpy().view(np.uint8).ravel()
    assert got.size == ref.size
    assert np.array_equal(got, ref)
    assert int(st.item()) == 0
