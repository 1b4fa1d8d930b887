"""fp64 oracle for the MoE layer — TEST INFRASTRUCTURE.

Only tests, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline legs may use it.

What the layer computes, per token t (page "3 ways to speed up MoE inference
on NVIDIA DGX Spark", §2: each MoE layer routes a token to 8 of 512 routed
experts plus one shared expert; §3: moe_intermediate_size 768; hidden size
2560 from the LM-head description in §2 and §4):

  1. router logits    l[t, e] = sum_j x[t, j] * Wr[e, j]          (+ bias)
  2. selection        S_t = the k experts with the largest key
                      key = fp32(logit + bias); ties -> lower expert index;
                      -0 is ranked as +0 and NaN as -inf
  3. weights          w[t, j] = exp(key_j - m) / sum_{i in S_t} exp(key_i - m)
                      (a softmax over all E, renormalised over the k selected,
                      is the same number)
  4. routed experts   h = silu(Wg x) * (Wu x),  silu(g) = g / (1 + e^-g)
                      out_e = Wd h
  5. output           y[t] = sum_j w[t, j] * out_{e_j}(x_t) + shared(x_t)
                      The shared expert enters with weight 1 (the pages give
                      no gate or scaling for it).

Readings taken where the pages are silent:
the router is a bias-free linear map unless a bias is supplied; a supplied
bias is added before both selection and weights; the softmax/top-k/renormalise
order is as above; the expert body is SwiGLU; there is no routed scaling
factor; the intermediate h is not rounded.

Index parity is decided on the GPU's own fp32 logits (both sides rank the same
fp32 numbers with the same fp32 bias addition), so ``route_topk`` accepts any
fp32 logits array.

Pins (tests/test_oracle_moe.py, tests/test_oracle_route.py): Sum w = 1; shift
invariance; k = E equals scipy's softmax; brute-force ranking with Python's
sort on small E with ties; one expert / identical experts equal a dense SwiGLU
FFN computed with torch float64 matmuls; a pure-Python triple loop on tiny
shapes; sort invariants against Python's sorted(); planted mistakes.
"""
from __future__ import annotations

import numpy as np

from . import mxfp4, mxfp8


def as_f64(t) -> np.ndarray:
    """torch tensor (any float dtype, incl. bf16) or array -> fp64 numpy, exactly."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            return t.detach().to("cpu").to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(t, dtype=np.float64)


def router_logits(x: np.ndarray, router_w: np.ndarray) -> np.ndarray:
    """l = x @ Wr^T in fp64 (x [T, d], Wr [E, d] hold bf16 values exactly)."""
    return as_f64(x) @ as_f64(router_w).T


def selection_keys(logits_f32: np.ndarray, bias=None) -> np.ndarray:
    """fp32 ranking keys: logit + bias added in fp32 (IEEE round-to-nearest-even).

    bias: None, [E] (broadcast to every token) or [T, E].
    """
    l32 = np.asarray(logits_f32, dtype=np.float32)
    if bias is None:
        return l32.copy()
    b = np.asarray(bias, dtype=np.float32)
    return (l32 + b).astype(np.float32)


def _rank_key(v: float) -> float:
    """Ranking value of one fp32 key: -0 ranks as +0 and NaN as -inf."""
    if np.isnan(v):
        return -np.inf
    return float(v) + 0.0


def route_topk(logits_f32: np.ndarray, k: int, bias=None):
    """Top-k selection and renormalised softmax weights.

    Returns (idx int32 [T, k] in descending key order, weights fp64 [T, k],
    keys fp32 [T, E]). Selection order: larger key first, equal keys -> lower
    expert index. Weights are a softmax over the k selected keys, in fp64.
    """
    keys = selection_keys(logits_f32, bias)
    T, E = keys.shape
    assert 1 <= k <= E
    idx = np.zeros((T, k), dtype=np.int32)
    wts = np.zeros((T, k), dtype=np.float64)
    for t in range(T):
        rk = np.array([_rank_key(v) for v in keys[t]], dtype=np.float64)
        order = np.lexsort((np.arange(E), -rk))      # primary: -rk ascending; then index
        sel = order[:k]
        idx[t] = sel
        kv = keys[t, sel].astype(np.float64)
        m = kv.max()
        ex = np.exp(kv - m)
        wts[t] = ex / ex.sum()
    return idx, wts, keys


def silu(g: np.ndarray) -> np.ndarray:
    return g / (1.0 + np.exp(-g))


def swiglu_ffn(x: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray, w_down: np.ndarray) -> np.ndarray:
    """Wd (silu(Wg x) * (Wu x)) for rows of x; all fp64.

    x [n, d], Wg/Wu [I, d], Wd [d, I] -> [n, d].
    """
    g = x @ w_gate.T
    u = x @ w_up.T
    return (silu(g) * u) @ w_down.T


class Expert:
    """One routed expert as fp64 dequantised weights (gate [I,d], up [I,d], down [d,I])."""

    def __init__(self, gate, up, down):
        self.gate, self.up, self.down = gate, up, down

    @classmethod
    def from_fp32(cls, gate_up_f32, down_f32):
        """Quantise fp32 weights with the oracle's MX rule and keep the exact values."""
        gu = mxfp4.fake_quantize(np.asarray(gate_up_f32, dtype=np.float32))
        dn = mxfp4.fake_quantize(np.asarray(down_f32, dtype=np.float32))
        I = gu.shape[0] // 2
        return cls(gu[:I], gu[I:], dn)


def expert_outputs(x_rows, gate_up_f32, down_f32, act_mxfp8: bool = False) -> np.ndarray:
    """One routed expert applied to some token rows, in fp64.

    The expert's fp32 weights (gate_up [2I, d], down [d, I]) are quantised
    with the MX rule (Expert.from_fp32), then out = Wd (silu(Wg x) * (Wu x))
    for every row of x_rows [n, d]. This is step 4 of the layer on its own,
    so that callers can evaluate many experts in separate processes and hand
    the results to moe_layer(expert_out=...).

    act_mxfp8: the 8-bit-activation (W4A8) mode — x is replaced by its MXFP8
    value (mxfp8.fake_quantize, per 32 along d) before the gate/up products,
    and h by its MXFP8 value (per 32 along I) before the down product; every
    product and sum is still exact fp64. Page "3 ways to speed up MoE
    inference on NVIDIA DGX Spark", §2 (the W4A8 baseline configuration).
    """
    e = Expert.from_fp32(gate_up_f32, down_f32)
    x = as_f64(x_rows)
    if not act_mxfp8:
        return swiglu_ffn(x, e.gate, e.up, e.down)
    xq = mxfp8.fake_quantize(x)
    h = silu(xq @ e.gate.T) * (xq @ e.up.T)
    return mxfp8.fake_quantize(h) @ e.down.T


def moe_layer(x, router_w, experts, shared, k: int, bias=None, idx=None, logits_f32=None,
              expert_out=None):
    """The whole layer in fp64.

    x          [T, d] (bf16 values)
    router_w   [E, d]
    experts    mapping expert id -> Expert (only the selected ones are needed)
    shared     (gate [I, d], up [I, d], down [d, I]) fp64, or None
    bias       None, [E] or [T, E]
    idx        optional [T, k] routing to use instead of the oracle's own
               (the GPU-reported indices, after they were checked)
    logits_f32 optional fp32 logits to rank; default: fp32(oracle fp64 logits)
    expert_out optional mapping (t, j) -> out_{idx[t, j]}(x_t) [d] from
               expert_outputs(); used instead of `experts` (which may then be
               None). The weights and the sum below are the same either way.

    Returns dict(logits fp64 [T,E], idx [T,k], weights fp64 [T,k], y fp64 [T,d]).
    Weights are computed from the oracle's fp64 logits (plus bias) at the
    selected indices.
    """
    x = as_f64(x)
    T, d = x.shape
    l64 = router_logits(x, router_w)
    if idx is None:
        l32 = l64.astype(np.float32) if logits_f32 is None else logits_f32
        idx, _, _ = route_topk(l32, k, bias)
    idx = np.asarray(idx)
    key64 = l64.copy()
    if bias is not None:
        key64 = key64 + np.broadcast_to(np.asarray(bias, dtype=np.float64), l64.shape)
    wts = np.zeros((T, k), dtype=np.float64)
    y = np.zeros((T, d), dtype=np.float64)
    for t in range(T):
        kv = key64[t, idx[t]]
        ex = np.exp(kv - kv.max())
        wts[t] = ex / ex.sum()
        for j in range(k):
            if expert_out is not None:
                out = np.asarray(expert_out[(t, j)], dtype=np.float64)
            else:
                ex_ = experts[int(idx[t, j])]
                out = swiglu_ffn(x[t:t + 1], ex_.gate, ex_.up, ex_.down)[0]
            y[t] += wts[t, j] * out
    if shared is not None:
        sg, su, sd = (as_f64(a) for a in shared)
        y += swiglu_ffn(x, sg, su, sd)
    return {"logits": l64, "idx": idx, "weights": wts, "y": y}


def sort_by_expert(idx: np.ndarray, E: int):
    """Group the (token, slot) pairs by expert, stable in p = t*k + j.

    Returns dict(counts int32 [E], offsets int32 [E+1] (exclusive scan),
    perm int32 [T*k] (sorted position -> p), inv int32 [T*k] (p -> sorted
    position), active int32 [D] (experts with count > 0, ascending), D).
    Page "MoE-SpeQ ...", §4.2: collect every draft token's expert assignment,
    sort by expert id, and run each expert once over its tokens.
    """
    flat = np.asarray(idx, dtype=np.int64).ravel()
    n = flat.size
    counts = np.bincount(flat, minlength=E).astype(np.int32)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    perm = np.zeros(n, dtype=np.int32)
    fill = offsets[:-1].copy()
    for p in range(n):                      # stable: visit p in increasing order
        e = flat[p]
        perm[fill[e]] = p
        fill[e] += 1
    inv = np.zeros(n, dtype=np.int32)
    inv[perm] = np.arange(n, dtype=np.int32)
    active = np.nonzero(counts)[0].astype(np.int32)
    return {"counts": counts, "offsets": offsets, "perm": perm, "inv": inv,
            "active": active, "D": int(active.size)}
