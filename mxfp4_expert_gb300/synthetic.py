"""Device layers built from the seeded synthetic workloads (for tests and benchmarks).

Weights are drawn by ``workloads`` (fp32 N(0, 0.02) experts, bf16 router and
shared expert) and packed on the GPU with ``moe_pack_mxfp4``. Nothing here
computes any part of the layer.
"""
from __future__ import annotations

import torch

import workloads as wl

from . import (MOE_LAYOUT_TILE16, MOE_LAYOUT_TILE16_GATEUP, Layer, moe_describe_packed,
               moe_pack_mxfp4)


def build_layer(w: wl.Workload, set_idx: int = 0, device="cuda", chunk: int = 32,
                dev_status: torch.Tensor | None = None) -> Layer:
    """Draw set `set_idx` of workload `w` on `device` and pack its experts."""
    router = wl.gen_router(w, set_idx, device)
    shared = wl.gen_shared(w, set_idx, device)
    gu_desc = moe_describe_packed(w.E, 2 * w.I, w.d, MOE_LAYOUT_TILE16_GATEUP)
    dn_desc = moe_describe_packed(w.E, w.d, w.I, MOE_LAYOUT_TILE16)
    gu = torch.empty(gu_desc.total_bytes, dtype=torch.uint8, device=device)
    dn = torch.empty(dn_desc.total_bytes, dtype=torch.uint8, device=device)
    bg, bd = gu_desc.bytes_per_mat, dn_desc.bytes_per_mat
    for e0 in range(0, w.E, chunk):
        n = min(chunk, w.E - e0)
        gu_f, dn_f = wl.gen_experts(w, set_idx, e0, n, device)
        moe_pack_mxfp4(gu_f, MOE_LAYOUT_TILE16_GATEUP, out=gu[e0 * bg:(e0 + n) * bg], dev_status=dev_status)
        moe_pack_mxfp4(dn_f, MOE_LAYOUT_TILE16, out=dn[e0 * bd:(e0 + n) * bd], dev_status=dev_status)
        del gu_f, dn_f
    return Layer(router, gu, gu_desc, dn, dn_desc, *shared, top_k=w.k)


def clone_rotated(base: Layer, w: wl.Workload, set_idx: int, device="cuda") -> Layer:
    """A further weight set for L2-defeating cycles, cheap to make.

    Router and shared expert are drawn fresh for `set_idx`; the packed routed
    experts are set 0's, rotated by 16*set_idx experts and copied to new memory
    (so no two sets share an address). Drawing 12 GB of fp32 per set would
    dominate a benchmark's run time; the bytes each call reads are the same.
    """
    router = wl.gen_router(w, set_idx, device)
    shared = wl.gen_shared(w, set_idx, device)
    r = (16 * set_idx) % w.E
    bg, bd = base.struct.gate_up_desc.bytes_per_mat, base.struct.down_desc.bytes_per_mat
    gu = torch.roll(base.gate_up, shifts=r * bg)
    dn = torch.roll(base.down, shifts=r * bd)
    return Layer(router, gu, base.struct.gate_up_desc, dn, base.struct.down_desc, *shared, top_k=w.k)


def inputs(w: wl.Workload, set_idx: int = 0, device="cuda"):
    """(x bf16 [T, d], bias fp32 or None) for one call."""
    return wl.gen_x(w, set_idx, device), wl.gen_bias(w, set_idx, device)
