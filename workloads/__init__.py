"""Seeded synthetic inputs for the MXFP4 mixture-of-experts layer.

This module only draws random numbers with the shapes, value distributions and
routing structure of the layer's workloads. It holds none of the layer's
arithmetic: no quantisation, no routing, no expert math. Both the fp64 oracle
(test infrastructure) and the CUDA path receive their inputs from here; neither
side generates inputs of its own.

Workloads (shapes from the page "3 ways to speed up MoE inference on NVIDIA
DGX Spark", §2 and §3: 512 routed experts, top-8, one shared expert,
hidden size 2560, moe_intermediate_size 768; the 4-token verify window and the
"up to 32 experts" it touches are from §5 of the same page):

  tiny         T=1,    d=512,  E=32,  k=4, I=128, 1 weight set
  ling_t1      T=1,    d=2560, E=512, k=8, I=768, 32 weight sets (cycled)
  mtp_t4       T=4,    Ling shapes, 32 sets; per-token bias picks 8..32 experts
  zipf_t64     T=64,   Ling shapes, 16 sets; bias gives Zipf(1.1) popularity
  prefill_t4096 T=4096, Ling shapes, 1 set; natural (near-uniform) routing

Value distributions: expert weights fp32 N(0, 0.02); router and shared-expert
weights N(0, 0.02) rounded to bf16; activations bf16 N(0, 1).

Seeding: every tensor has its own sub-seed derived from (seed, set, tensor id,
expert), so any single expert can be regenerated on its own. Tensors are drawn
with torch's generator on the device given; the same seed on the same device
type gives the same values. Large weight sets are drawn on the GPU; the oracle
then receives copies of exactly those tensors.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

__all__ = [
    "Workload", "WORKLOADS", "get", "sub_seed",
    "gen_x", "gen_router", "gen_shared", "gen_expert", "gen_bias",
    "mtp_expert_sets", "ZIPF_S", "ZIPF_ALPHA", "WEIGHT_STD",
]

WEIGHT_STD = 0.02
ZIPF_S = 1.1
# Scale of the log-popularity bias for the T=64 workload. Chosen once with
# calibrate_zipf_alpha(): with router logits of standard deviation ~1.01
# (x ~ N(0,1), W_r ~ N(0,0.02), d=2560), alpha=0.52 makes the log-log slope
# of selection frequency against popularity rank (ranks 2..128) equal -1.1,
# and gives about 150 distinct experts per 64-token batch.
ZIPF_ALPHA = 0.52

# tensor ids for sub-seeds
_TID = {"x": 1, "router": 2, "shared_gate": 3, "shared_up": 4, "shared_down": 5,
        "expert": 6, "bias": 7, "mtp": 8}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    I: int
    E: int
    k: int
    sets: int
    routing: str          # "natural" | "mtp" | "zipf"
    seed: int = 0

    @property
    def has_bias(self) -> bool:
        return self.routing in ("mtp", "zipf")

    @property
    def bias_row_stride(self) -> int:
        """0: one bias row [E] shared by all tokens; E: one row per token."""
        return self.E if self.routing == "mtp" else 0


WORKLOADS = {
    "tiny": Workload("tiny", T=1, d=512, I=128, E=32, k=4, sets=1, routing="natural"),
    "ling_t1": Workload("ling_t1", T=1, d=2560, I=768, E=512, k=8, sets=32, routing="natural"),
    "mtp_t4": Workload("mtp_t4", T=4, d=2560, I=768, E=512, k=8, sets=32, routing="mtp"),
    "zipf_t64": Workload("zipf_t64", T=64, d=2560, I=768, E=512, k=8, sets=16, routing="zipf"),
    "prefill_t4096": Workload("prefill_t4096", T=4096, d=2560, I=768, E=512, k=8, sets=1,
                              routing="natural"),
}


def get(name: str, **overrides) -> Workload:
    return dataclasses.replace(WORKLOADS[name], **overrides)


def sub_seed(w: Workload, set_idx: int, tensor: str, expert: int = 0) -> int:
    return (w.seed * 1000003 + set_idx * 131 + _TID[tensor] * 7919 + expert * 104729) % (2**63 - 1)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, std, seed, device, dtype=torch.float32):
    g = _gen(seed, device)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def gen_x(w: Workload, set_idx: int = 0, device="cpu", T: int | None = None) -> torch.Tensor:
    """Activations, bf16 [T, d], N(0, 1)."""
    T = w.T if T is None else T
    return _normal((T, w.d), 1.0, sub_seed(w, set_idx, "x"), device, torch.bfloat16)


def gen_router(w: Workload, set_idx: int = 0, device="cpu") -> torch.Tensor:
    """Router weight, bf16 [E, d], N(0, 0.02) rounded to bf16."""
    return _normal((w.E, w.d), WEIGHT_STD, sub_seed(w, set_idx, "router"), device, torch.bfloat16)


def gen_shared(w: Workload, set_idx: int = 0, device="cpu"):
    """Shared expert, bf16: gate [I, d], up [I, d], down [d, I]."""
    g = _normal((w.I, w.d), WEIGHT_STD, sub_seed(w, set_idx, "shared_gate"), device, torch.bfloat16)
    u = _normal((w.I, w.d), WEIGHT_STD, sub_seed(w, set_idx, "shared_up"), device, torch.bfloat16)
    dn = _normal((w.d, w.I), WEIGHT_STD, sub_seed(w, set_idx, "shared_down"), device, torch.bfloat16)
    return g, u, dn


def gen_expert(w: Workload, set_idx: int, expert: int, device="cpu"):
    """One routed expert before quantisation, fp32 N(0, 0.02).

    Returns (gate_up [2I, d], down [d, I]); rows 0..I-1 of gate_up are the
    gate projection, rows I..2I-1 the up projection.
    """
    seed = sub_seed(w, set_idx, "expert", expert)
    g = _gen(seed, device)
    gu = torch.randn((2 * w.I, w.d), generator=g, device=device, dtype=torch.float32).mul_(WEIGHT_STD)
    dn = torch.randn((w.d, w.I), generator=g, device=device, dtype=torch.float32).mul_(WEIGHT_STD)
    return gu, dn


def gen_experts(w: Workload, set_idx: int, first: int, count: int, device="cpu"):
    """Experts [first, first+count) stacked: gate_up [n, 2I, d], down [n, d, I]."""
    gus, dns = [], []
    for e in range(first, first + count):
        gu, dn = gen_expert(w, set_idx, e, device)
        gus.append(gu)
        dns.append(dn)
    return torch.stack(gus), torch.stack(dns)


def mtp_expert_sets(w: Workload, set_idx: int):
    """The 4-token verify workload: per-token expert sets with a seeded union size D.

    D is drawn from {8, 12, ..., 32}. D distinct experts are drawn; token 0
    takes the first 8, the remaining D-8 are split as evenly as possible over
    tokens 1..T-1, and each of those tokens fills up to 8 with experts already
    used by earlier tokens. The union over tokens is exactly D experts.
    Returns (D, list of T sorted lists of 8 expert ids).
    """
    rng = np.random.default_rng(sub_seed(w, set_idx, "mtp"))
    choices = list(range(w.k, min(w.T * w.k, w.E) + 1, 4))
    D = int(rng.choice(choices))
    pool = rng.permutation(w.E)[:D]
    sets = [list(pool[: w.k])]
    fresh = list(pool[w.k:])
    n_rest = w.T - 1
    shares = [len(fresh) // n_rest + (1 if i < len(fresh) % n_rest else 0) for i in range(n_rest)]
    pos = 0
    for i in range(n_rest):
        new = fresh[pos: pos + shares[i]]
        pos += shares[i]
        used = sorted(set().union(*[set(s) for s in sets]))
        need = w.k - len(new)
        old = list(rng.choice(used, size=need, replace=False)) if need > 0 else []
        sets.append(list(new) + old)
    return D, [sorted(int(e) for e in s) for s in sets]


def gen_bias(w: Workload, set_idx: int = 0, device="cpu"):
    """Router bias (fp32) for the biased workloads, or None.

    mtp:  [T, E]; +16 on each token's 8 experts, 0 elsewhere (logits have
          standard deviation ~1, so those 8 are the top-8; adding the same
          constant keeps their relative softmax weights).
    zipf: [E]; b[e] = ZIPF_ALPHA * ln p(rank(e)), p(r) ~ r^-1.1 over ranks
          1..E, ranks assigned by a seeded permutation.
    """
    if w.routing == "mtp":
        _, sets = mtp_expert_sets(w, set_idx)
        b = torch.zeros((w.T, w.E), dtype=torch.float32)
        for t, s in enumerate(sets):
            b[t, s] = 16.0
        return b.to(device)
    if w.routing == "zipf":
        rng = np.random.default_rng(sub_seed(w, set_idx, "bias"))
        rank = rng.permutation(w.E)                  # expert e has popularity rank rank[e]
        r = np.arange(1, w.E + 1, dtype=np.float64)
        p = r ** (-ZIPF_S)
        p /= p.sum()
        b = (ZIPF_ALPHA * np.log(p[rank])).astype(np.float32)
        return torch.from_numpy(b).to(device)
    return None


def calibrate_zipf_alpha(alphas=(0.5, 0.52, 0.54), trials=400, logit_std=1.01, seed=1):
    """Re-derive ZIPF_ALPHA: log-log slope of selection frequency vs rank per alpha.

    Uses independent N(0, logit_std^2) logits as a stand-in for x @ W_r^T and
    a plain argpartition for the top-k pick; this is a workload-shaping aid,
    not part of either implementation.
    """
    E, k, T = 512, 8, 64
    r = np.arange(1, E + 1)
    p = r ** -ZIPF_S
    p = p / p.sum()
    out = {}
    for a in alphas:
        rng = np.random.default_rng(seed)
        cnt = np.zeros(E)
        for _ in range(trials):
            rank = rng.permutation(E)
            logits = rng.standard_normal((T, E)) * logit_std + a * np.log(p[rank])
            top = np.argpartition(-logits, k, axis=1)[:, :k]
            np.add.at(cnt, rank[top.ravel()], 1)
        f = cnt / cnt.sum()
        out[a] = float(np.polyfit(np.log(r[1:128]), np.log(f[1:128] + 1e-12), 1)[0])
    return out


def weight_bytes(w: Workload, distinct_experts: int) -> int:
    """Algorithmic weight bytes read by one layer call.

    router E*d*2 + shared 3*d*I*2 + D*(3*d*I/2 codes + 3*d*I/32 scales).
    """
    per_expert = 3 * w.d * w.I // 2 + 3 * w.d * w.I // 32
    return w.E * w.d * 2 + 3 * w.d * w.I * 2 + distinct_experts * per_expert


def layer_flops(w: Workload, distinct_slots: int) -> int:
    """Multiply-add work (2 flops each) of one call: router, shared, routed slots."""
    T = w.T
    return 2 * (T * w.E * w.d + T * 3 * w.d * w.I + distinct_slots * 3 * w.d * w.I)
