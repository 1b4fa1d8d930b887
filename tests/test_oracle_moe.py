"""Pins for the layer oracle: dense special cases via torch float64 (a library
routine), a pure-Python triple loop on tiny shapes, and planted mistakes."""
import math
import os

import numpy as np
import pytest
import torch

import workloads
from oracle import moe, mxfp4


def torch_dense_swiglu(x, g, u, d):
    X, G, U, Dn = (torch.from_numpy(np.asarray(a, dtype=np.float64)) for a in (x, g, u, d))
    return (torch.nn.functional.silu(X @ G.T) * (X @ U.T) @ Dn.T).numpy()


def small_layer(seed=0, T=3, d=64, I=32, E=8, k=2):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d))
    wr = rng.standard_normal((E, d)) * 0.1
    experts = {}
    for e in range(E):
        gu = (rng.standard_normal((2 * I, d)) * 0.05).astype(np.float32)
        dn = (rng.standard_normal((d, I)) * 0.05).astype(np.float32)
        experts[e] = moe.Expert.from_fp32(gu, dn)
    shared = tuple(rng.standard_normal(s) * 0.05 for s in [(I, d), (I, d), (d, I)])
    return x, wr, experts, shared


def triple_loop_layer(x, wr, experts, shared, k):
    """Pure-Python loops, no numpy arithmetic."""
    T, d = len(x), len(x[0])
    E = len(wr)
    y = [[0.0] * d for _ in range(T)]
    for t in range(T):
        logits = [sum(float(x[t][j]) * float(wr[e][j]) for j in range(d)) for e in range(E)]
        sel = sorted(range(E), key=lambda e: (-logits[e], e))[:k]
        m = max(logits[e] for e in sel)
        z = sum(math.exp(logits[e] - m) for e in sel)
        mats = [(math.exp(logits[e] - m) / z, experts[e].gate, experts[e].up, experts[e].down)
                for e in sel] + [(1.0,) + tuple(shared)]
        for wgt, G, U, Dn in mats:
            I = len(G)
            h = []
            for i in range(I):
                g = sum(float(G[i][j]) * float(x[t][j]) for j in range(d))
                u = sum(float(U[i][j]) * float(x[t][j]) for j in range(d))
                h.append(g / (1.0 + math.exp(-g)) * u)
            for r in range(d):
                y[t][r] += wgt * sum(float(Dn[r][i]) * h[i] for i in range(I))
    return np.array(y)


def test_layer_matches_triple_loop():
    x, wr, experts, shared = small_layer()
    out = moe.moe_layer(x, wr, experts, shared, k=2)
    ref = triple_loop_layer(x, wr, experts, shared, k=2)
    assert np.allclose(out["y"], ref, rtol=1e-11, atol=1e-12)


def test_one_expert_top1_is_dense_ffn_plus_shared():
    x, wr, experts, shared = small_layer(seed=1, E=1, k=1)
    out = moe.moe_layer(x, wr, experts, shared, k=1)
    e = experts[0]
    ref = torch_dense_swiglu(x, e.gate, e.up, e.down) + torch_dense_swiglu(x, *shared)
    assert np.allclose(out["weights"], 1.0)
    assert np.allclose(out["y"], ref, rtol=1e-12, atol=1e-13)


def test_identical_experts_collapse_to_dense():
    x, wr, experts, shared = small_layer(seed=2, E=8, k=3)
    same = {e: experts[0] for e in range(8)}
    out = moe.moe_layer(x, wr, same, None, k=3)
    ref = torch_dense_swiglu(x, experts[0].gate, experts[0].up, experts[0].down)
    assert np.allclose(out["y"], ref, rtol=1e-12, atol=1e-13)


def test_supplied_idx_and_bias():
    x, wr, experts, shared = small_layer(seed=3, E=8, k=2)
    bias = np.zeros(8, dtype=np.float32)
    bias[5] = 50.0
    out = moe.moe_layer(x, wr, experts, shared, k=2, bias=bias)
    assert np.all(out["idx"][:, 0] == 5)
    out2 = moe.moe_layer(x, wr, experts, shared, k=2, bias=bias, idx=out["idx"])
    assert np.array_equal(out["y"], out2["y"])


def test_experts_from_fp32_use_the_mx_values():
    rng = np.random.default_rng(4)
    gu = (rng.standard_normal((64, 64)) * 0.02).astype(np.float32)
    dn = (rng.standard_normal((64, 32)) * 0.02).astype(np.float32)
    e = moe.Expert.from_fp32(gu, dn)
    assert np.array_equal(np.vstack([e.gate, e.up]), mxfp4.fake_quantize(gu))
    assert np.array_equal(e.down, mxfp4.fake_quantize(dn))


def test_expert_outputs_path_matches_triple_loop():
    """moe_layer(expert_out=...) with per-(token, slot) outputs from
    expert_outputs() gives the triple loop's layer (the path the full-size
    GPU parity checks use to spread the oracle over processes)."""
    rng = np.random.default_rng(6)
    T, d, I, E, k = 3, 64, 32, 8, 2
    x = rng.standard_normal((T, d))
    wr = rng.standard_normal((E, d)) * 0.1
    raw = {e: ((rng.standard_normal((2 * I, d)) * 0.05).astype(np.float32),
               (rng.standard_normal((d, I)) * 0.05).astype(np.float32)) for e in range(E)}
    experts = {e: moe.Expert.from_fp32(*raw[e]) for e in range(E)}
    shared = tuple(rng.standard_normal(s) * 0.05 for s in [(I, d), (I, d), (d, I)])
    idx = moe.moe_layer(x, wr, experts, shared, k=k)["idx"]
    outs = {}
    for e in set(idx.ravel().tolist()):
        pairs = [(t, j) for t in range(T) for j in range(k) if idx[t, j] == e]
        rows = moe.expert_outputs(x[[t for t, _ in pairs]], *raw[e])
        outs.update({p: rows[i] for i, p in enumerate(pairs)})
    out = moe.moe_layer(x, wr, None, shared, k=k, idx=idx, expert_out=outs)
    ref = triple_loop_layer(x, wr, experts, shared, k=k)
    assert np.allclose(out["y"], ref, rtol=1e-11, atol=1e-12)
    # a wrong pairing (slots of one token swapped) is visible
    bad = dict(outs)
    bad[(0, 0)], bad[(0, 1)] = outs[(0, 1)], outs[(0, 0)]
    wrong = moe.moe_layer(x, wr, None, shared, k=k, idx=idx, expert_out=bad)["y"]
    assert _rel(wrong, ref) > 1e-3


def _loops_w4a8(x, gu, dn, quant):
    """Pure-Python loops for one expert in the MXFP8-activation mode; the only
    library calls are the pinned quantisers (mxfp4 for the weights, `quant`
    for the activations)."""
    G, U, Dn = (mxfp4.fake_quantize(m) for m in (gu[: len(gu) // 2], gu[len(gu) // 2:], dn))
    xq = quant(x)
    out = []
    for t in range(len(x)):
        h = []
        for i in range(len(G)):
            g = sum(float(G[i][j]) * float(xq[t][j]) for j in range(len(x[0])))
            u = sum(float(U[i][j]) * float(xq[t][j]) for j in range(len(x[0])))
            h.append(g / (1.0 + math.exp(-g)) * u)
        hq = quant(np.array([h]))[0]
        out.append([sum(float(Dn[r][i]) * float(hq[i]) for i in range(len(h))) for r in range(len(Dn))])
    return np.array(out)


def test_expert_outputs_w4a8_matches_loops():
    """The MXFP8-activation mode quantises x before gate/up and h before down,
    nothing else; planted variants (only x, only h, neither) are caught."""
    from oracle import mxfp8
    rng = np.random.default_rng(8)
    T, d, I = 3, 64, 32
    x = rng.standard_normal((T, d))
    gu = (rng.standard_normal((2 * I, d)) * 0.05).astype(np.float32)
    dn = (rng.standard_normal((d, I)) * 0.05).astype(np.float32)
    got = moe.expert_outputs(x, gu, dn, act_mxfp8=True)
    ref = _loops_w4a8(x, gu, dn, mxfp8.fake_quantize)
    assert np.allclose(got, ref, rtol=1e-11, atol=1e-12)
    ident = lambda a: np.asarray(a, dtype=np.float64)   # noqa: E731
    plain = moe.expert_outputs(x, gu, dn)
    assert np.allclose(plain, _loops_w4a8(x, gu, dn, ident), rtol=1e-11, atol=1e-12)
    only_x = _loops_w4a8(x, gu, dn, lambda a: mxfp8.fake_quantize(a) if np.shape(a)[1] == d else ident(a))
    only_h = _loops_w4a8(x, gu, dn, lambda a: mxfp8.fake_quantize(a) if np.shape(a)[1] == I else ident(a))
    for bad in (plain, only_x, only_h):
        assert _rel(bad, got) > 1e-3


# planted mistakes: each plausible bug must change the result beyond tolerance ----

def _rel(a, b):
    return np.linalg.norm(a - b) / np.linalg.norm(b)


def test_planted_mistakes_are_caught():
    x, wr, experts, shared = small_layer(seed=5, E=8, k=2)
    ref = torch_dense_swiglu  # noqa: F841  (documentation of the library pin used above)
    good = triple_loop_layer(x, wr, experts, shared, k=2)
    # (a) shared expert dropped
    no_shared = moe.moe_layer(x, wr, experts, (np.zeros_like(shared[0]), shared[1], shared[2]), k=2)["y"]
    # (b) gate and up swapped in every expert
    swapped = {e: moe.Expert(v.up, v.gate, v.down) for e, v in experts.items()}
    sw = moe.moe_layer(x, wr, swapped, shared, k=2)["y"]
    # (c) down projection transposed-by-mistake is shape-incompatible unless square; use d=I
    for bad in (no_shared, sw):
        assert _rel(bad, good) > 1e-3


def test_workload_shapes_match_golden_facts():
    facts = {}
    with open(os.path.join(os.path.dirname(__file__), "golden", "ling_moe_shape.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split("=")
                facts[k.strip()] = int(v)
    w = workloads.WORKLOADS["ling_t1"]
    assert (w.E, w.k, w.I, w.d) == (facts["routed_experts"], facts["top_k"],
                                     facts["moe_intermediate_size"], facts["hidden_size"])
    assert facts["shared_experts"] == 1
    assert workloads.WORKLOADS["mtp_t4"].T == facts["verify_tokens"]
    assert min(workloads.WORKLOADS["mtp_t4"].T * 8, 512) == facts["verify_max_experts"]
