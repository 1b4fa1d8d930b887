"""Pins for the routing oracle (top-k + renormalised softmax + expert sort)."""
import numpy as np
import pytest
import scipy.special

from oracle import moe


def brute_rank(keys_row, k):
    """Python's sort on (-value, index), with -0 -> +0 and NaN -> -inf."""
    def val(v):
        v = float(v)
        return float("-inf") if v != v else v + 0.0
    order = sorted(range(len(keys_row)), key=lambda e: (-val(keys_row[e]), e))
    return order[:k]


def test_weights_sum_to_one_and_shift_invariance():
    rng = np.random.default_rng(0)
    # multiples of 2^-10 in [-8, 8]: adding 1.0 in fp32 is exact, so ranking is unchanged
    logits = (rng.integers(-8192, 8192, (16, 64)) / 1024.0).astype(np.float32)
    idx, w, _ = moe.route_topk(logits, 8)
    assert np.all(np.abs(w.sum(1) - 1.0) <= 1e-12)
    idx2, w2, _ = moe.route_topk(logits + np.float32(1.0), 8)
    assert np.array_equal(idx, idx2)
    assert np.allclose(w, w2, rtol=0, atol=1e-12)


def test_k_equals_E_is_full_softmax():
    rng = np.random.default_rng(1)
    logits = rng.standard_normal((5, 32)).astype(np.float32)
    idx, w, _ = moe.route_topk(logits, 32)
    ref = scipy.special.softmax(logits.astype(np.float64), axis=1)
    for t in range(5):
        assert np.allclose(w[t], ref[t, idx[t]], rtol=1e-13, atol=0)
        assert sorted(idx[t].tolist()) == list(range(32))


def test_topk_equals_renormalised_full_softmax():
    rng = np.random.default_rng(2)
    logits = rng.standard_normal((7, 512)).astype(np.float32)
    idx, w, _ = moe.route_topk(logits, 8)
    full = scipy.special.softmax(logits.astype(np.float64), axis=1)
    for t in range(7):
        sel = full[t, idx[t]]
        assert np.allclose(w[t], sel / sel.sum(), rtol=1e-12, atol=0)


def test_bruteforce_ranking_with_ties_signed_zero_and_nan():
    rng = np.random.default_rng(3)
    for trial in range(200):
        E = int(rng.integers(2, 24))
        k = int(rng.integers(1, E + 1))
        vals = rng.choice(np.array([-1.0, -0.0, 0.0, 0.5, 0.5, 2.0, np.nan, -np.inf, 3.0],
                                   dtype=np.float32), size=(1, E))
        idx, _, _ = moe.route_topk(vals, k)
        assert idx[0].tolist() == brute_rank(vals[0], k), (vals, k)


def test_bias_broadcast_and_per_token():
    rng = np.random.default_rng(4)
    logits = rng.standard_normal((3, 16)).astype(np.float32)
    b = rng.standard_normal(16).astype(np.float32)
    i1, w1, _ = moe.route_topk(logits, 4, b)
    i2, w2, _ = moe.route_topk(logits, 4, np.broadcast_to(b, (3, 16)))
    i3, _, _ = moe.route_topk((logits + b).astype(np.float32), 4)
    assert np.array_equal(i1, i2) and np.array_equal(i1, i3) and np.allclose(w1, w2)
    for t in range(3):
        assert i1[t].tolist() == brute_rank((logits[t] + b), 4)


def test_sort_by_expert_matches_python_sorted():
    rng = np.random.default_rng(5)
    for T, E, k in [(1, 512, 8), (4, 512, 8), (64, 512, 8), (13, 8, 3), (1, 4, 4)]:
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        r = moe.sort_by_expert(idx, E)
        pairs = sorted((int(idx.ravel()[p]), p) for p in range(T * k))
        assert r["perm"].tolist() == [p for _, p in pairs]
        assert np.array_equal(r["inv"][r["perm"]], np.arange(T * k))
        assert r["counts"].sum() == T * k and r["offsets"][-1] == T * k
        assert r["active"].tolist() == sorted(set(idx.ravel().tolist()))
        for e in range(E):
            seg = r["perm"][r["offsets"][e]:r["offsets"][e + 1]]
            assert all(idx.ravel()[p] == e for p in seg)


# planted mistakes -------------------------------------------------------------

def test_planted_ties_to_higher_index_is_caught():
    vals = np.array([[1.0, 2.0, 2.0, 0.0]], dtype=np.float32)
    idx, _, _ = moe.route_topk(vals, 2)
    assert idx[0].tolist() == [1, 2]
    wrong = np.argsort(-vals[0], kind="stable")[::-1][:2]          # a plausible bug
    assert wrong.tolist() != brute_rank(vals[0], 2)


def test_planted_unrenormalised_weights_are_caught():
    rng = np.random.default_rng(6)
    logits = rng.standard_normal((4, 64)).astype(np.float32)
    idx, w, _ = moe.route_topk(logits, 8)
    full = scipy.special.softmax(logits.astype(np.float64), axis=1)
    unnorm = np.take_along_axis(full, idx.astype(np.int64), 1)
    assert not np.all(np.abs(unnorm.sum(1) - 1.0) <= 1e-12)      # the Sum w = 1 pin rejects it
    assert np.all(np.abs(w.sum(1) - 1.0) <= 1e-12)
