"""moe_route_topk and moe_sort_by_expert on the GPU vs. the oracle.

Indices, counts, offsets, permutations: bit-exact (the oracle ranks the same
fp32 logits with the same fp32 bias addition). Weights: fp32 exp vs fp64,
|w_gpu - w_ref| <= 2e-6 and |sum w - 1| <= 2e-6.
"""
import numpy as np
import pytest
import torch

from oracle import moe as omoe

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    import mxfp4_expert_gb300 as mx
    return mx


def make_logits(T, E, seed, ties=False, specials=False):
    rng = np.random.default_rng(seed)
    l = rng.standard_normal((T, E)).astype(np.float32)
    if ties:
        l = (np.round(l * 4) / 4).astype(np.float32)
    if specials:
        m = rng.random((T, E))
        l[m < 0.05] = -0.0
        l[(m >= 0.05) & (m < 0.1)] = 0.0
        l[(m >= 0.1) & (m < 0.12)] = np.nan
        l[(m >= 0.12) & (m < 0.14)] = -np.inf
    return l


def check_route(mx, l, k, bias=None):
    T, E = l.shape
    lt = torch.from_numpy(l).cuda()
    bt = None if bias is None else torch.from_numpy(bias).cuda()
    idx, w = mx.moe_route_topk(lt, k, bt)
    torch.cuda.synchronize()
    ri, rw, _ = omoe.route_topk(l, k, bias)
    gi = idx.cpu().numpy()
    assert np.array_equal(gi, ri)
    gw = w.cpu().numpy().astype(np.float64)
    fin = np.isfinite(rw).all(axis=1)
    assert np.all(np.abs(gw[fin] - rw[fin]) <= 2e-6)
    assert np.all(np.abs(gw[fin].sum(1) - 1.0) <= 2e-6)


@pytest.mark.parametrize("T,E,k", [(1, 512, 8), (4, 512, 8), (64, 512, 8), (3, 32, 4), (5, 40, 32),
                                   (7, 100, 3), (2, 1024, 32), (9, 1, 1), (33, 96, 8)])
def test_topk_random(mx, T, E, k):
    check_route(mx, make_logits(T, E, T * 1000 + E), k)


@pytest.mark.parametrize("T,E,k", [(16, 512, 8), (8, 32, 4), (4, 64, 32)])
def test_topk_ties_and_specials(mx, T, E, k):
    check_route(mx, make_logits(T, E, 7, ties=True), k)
    l = make_logits(T, E, 8, ties=True, specials=True)
    # keep at least k finite candidates per row so weights are defined
    check_route(mx, l, min(k, 4))


def test_topk_bias_broadcast_and_per_token(mx):
    l = make_logits(6, 512, 11)
    b = (np.random.default_rng(12).standard_normal(512) * 2).astype(np.float32)
    check_route(mx, l, 8, b)
    bt = (np.random.default_rng(13).standard_normal((6, 512)) * 2).astype(np.float32)
    check_route(mx, l, 8, bt)


def distinct_idx(T, E, k, seed):
    rng = np.random.default_rng(seed)
    return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,E,k", [(1, 512, 8), (4, 512, 8), (64, 512, 8), (130, 512, 8),
                                   (4096, 512, 8), (3, 32, 4), (300, 7, 7), (129, 1024, 32)])
def test_sort_by_expert_bit_exact(mx, T, E, k):
    idx = distinct_idx(T, E, k, T + E + k)
    r = mx.moe_sort_by_expert(torch.from_numpy(idx).cuda(), E)
    torch.cuda.synchronize()
    ref = omoe.sort_by_expert(idx, E)
    for key in ("counts", "offsets", "perm", "inv"):
        assert np.array_equal(r[key].cpu().numpy(), ref[key]), key
    D = int(r["n_active"].item())
    assert D == ref["D"]
    assert np.array_equal(r["active"].cpu().numpy()[:D], ref["active"])


def test_sort_flags_out_of_range_and_repeats(mx):
    idx = np.array([[0, 5, 5], [2, -1, 9], [1, 2, 3]], dtype=np.int32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    r = mx.moe_sort_by_expert(torch.from_numpy(idx).cuda(), 8, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & mx.DEV_INDEX_OOB
    inv = r["inv"].cpu().numpy()
    assert inv[2] == -1 and inv[4] == -1 and inv[5] == -1
    kept = [0, 1, 3, 6, 7, 8]
    ref = omoe.sort_by_expert(idx.ravel()[kept][:, None], 8)
    perm = r["perm"].cpu().numpy()[: len(kept)]
    assert [kept.index(p) for p in perm] == ref["perm"].tolist()
