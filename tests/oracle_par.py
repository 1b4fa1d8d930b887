"""Reference outputs of the fp64 oracle for the GPU parity tests (test infrastructure).

The full-size workloads route tokens to hundreds of distinct experts, and the
oracle quantises every one of them from its fp32 weights (about half a
second per Ling-shape expert). `reference_layer` therefore evaluates the
experts in a pool of worker processes (spawn context, so it is safe after
CUDA has been initialised in this process) with `oracle.moe.expert_outputs`
and lets `oracle.moe.moe_layer` combine the results. Expert weights come from
the seeded generators on the same device the library's layer was drawn on.

Also the per-element tolerance of a bf16 output: `bf16_rne` rounds fp64 to
the nearest bf16 value (ties to even), the best any bf16 result can do.
"""
from __future__ import annotations

import atexit
import multiprocessing as mp
import os

import numpy as np

import workloads as wl
from oracle import moe as omoe

_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        n = max(1, min(16, (os.cpu_count() or 2) - 1))
        _POOL = mp.get_context("spawn").Pool(n)
        atexit.register(_POOL.terminate)
    return _POOL


def reference_layer(w, set_idx, x_rows, router, shared, bias_rows, idx, device="cuda", act_mxfp8=False):
    """oracle.moe.moe_layer for the given token rows at the given (already
    checked) routing, with the experts evaluated in parallel processes.

    x_rows [n, d] (torch bf16 on the CPU), idx [n, k] int; act_mxfp8: the
    oracle's 8-bit-activation mode for the routed experts. Returns moe_layer's dict.
    """
    idx = np.asarray(idx)
    n, k = idx.shape
    xs = omoe.as_f64(x_rows)
    pairs_of = {}
    for t in range(n):
        for j in range(k):
            pairs_of.setdefault(int(idx[t, j]), []).append((t, j))
    experts = sorted(pairs_of)
    jobs = []
    for e in experts:
        gu, dn = wl.gen_expert(w, set_idx, e, device)
        rows = xs[[t for t, _ in pairs_of[e]]]
        jobs.append((rows, gu.cpu().numpy(), dn.cpu().numpy(), act_mxfp8))
    if len(jobs) > 4:
        results = _pool().starmap(omoe.expert_outputs, jobs, chunksize=1)
    else:
        results = [omoe.expert_outputs(*j) for j in jobs]
    outs = {}
    for e, res in zip(experts, results):
        for i, p in enumerate(pairs_of[e]):
            outs[p] = res[i]
    return omoe.moe_layer(xs, router, None, shared, k, bias=bias_rows, idx=idx, expert_out=outs)


def bf16_rne(v):
    """fp64 -> nearest bf16 value (8 significant bits, ties to even), as fp64.

    Normal range: the quantum at |v| in [2^(e-1), 2^e) is 2^(e-8); below
    2^-126 bf16 is subnormal with quantum 2^-133.
    """
    v = np.asarray(v, dtype=np.float64)
    _, e = np.frexp(v)
    q_exp = np.maximum(e.astype(np.int64) - 8, -133)
    q = np.ldexp(1.0, q_exp)
    return np.rint(v / q) * q


def bf16_ulp(v):
    """Spacing of bf16 numbers at |v| (0 at v = 0)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 7), 0.0)
