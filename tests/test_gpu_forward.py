"""moe_forward on the GPU vs. the fp64 oracle.

Per call: (1) the GPU's router logits are within 1e-5 * sum_j |x_j Wr_j| of
the oracle's fp64 logits; (2) the GPU's indices equal the oracle's ranking of
the GPU's own fp32 logits (plus bias) and the weights agree to 2e-6;
(3) y (bf16) against the oracle's fp64 layer output computed with those
indices: relative L2 <= 5e-3 and max |err| <= 2e-2 * rms(y_ref) per element.
The one exception to the per-element bound is an element whose GPU value is
exactly y_ref rounded to the nearest bf16 (no bf16 output can be closer);
such elements are counted, and the Ling-shape workloads require none.
Workloads are checked on every token, except prefill (T = 4096), which is
checked on at least 256 tokens chosen so that every expert is some checked
token's choice.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle_par
import workloads as wl
from oracle import moe as omoe

pytestmark = pytest.mark.gpu

REL_L2 = 5e-3
MAX_ABS = 2e-2


@pytest.fixture(scope="module")
def mx():
    import mxfp4_expert_gb300 as mx
    return mx


def run(mx, layer, x, bias, T, E, k):
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = mx.moe_forward(layer, x, bias, logits_out=logits, idx_out=idx, w_out=w, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return y, logits, idx, w


def check_layer(w, set_idx, layer, x, bias, out, tokens=None, device="cuda", strict=False):
    """Checks (1)-(3) on `tokens` (default: all). Returns (rel-L2, max|err|/rms,
    elements that needed the bf16-rounding exception); strict=True requires none."""
    y, logits, idx, wts = out
    tokens = list(range(w.T)) if tokens is None else list(tokens)
    xs = x[tokens].cpu()
    router = wl.gen_router(w, set_idx, device).cpu()
    gl = logits.cpu().numpy()[tokens]
    gi = idx.cpu().numpy()[tokens]
    b = None
    if bias is not None:
        b = bias.cpu().numpy()
        if b.ndim == 2:
            b = b[tokens]
    # (1) logits
    ref_l = omoe.router_logits(xs, router)
    bound = 1e-5 * (np.abs(omoe.as_f64(xs)) @ np.abs(omoe.as_f64(router)).T)
    assert np.all(np.abs(gl - ref_l) <= bound + 1e-30)
    # (2) routing from the GPU's own fp32 logits
    ri, rw, _ = omoe.route_topk(gl, w.k, b)
    assert np.array_equal(gi, ri)
    assert np.all(np.abs(wts.cpu().numpy()[tokens] - rw) <= 2e-6)
    # (3) y with the oracle's expert values at those indices
    shared = tuple(t.cpu() for t in wl.gen_shared(w, set_idx, device))
    if not layer.shape.has_shared:
        shared = None
    ref = oracle_par.reference_layer(w, set_idx, xs, router, shared, b, gi, device)
    yg = y.float().cpu().numpy().astype(np.float64)[tokens]
    yr = ref["y"]
    rel = np.linalg.norm(yg - yr) / np.linalg.norm(yr)
    rms = np.sqrt(np.mean(yr ** 2))
    err = np.abs(yg - yr)
    assert rel <= REL_L2, rel
    within = err <= MAX_ABS * rms
    rounded = yg == oracle_par.bf16_rne(yr)
    bad = ~(within | rounded)
    assert not bad.any(), (int(bad.sum()), float(err.max() / rms))
    n_exc = int(np.sum(~within))
    if strict:
        assert n_exc == 0, n_exc
    print(f"{w.name} set {set_idx}: {len(tokens)} tokens, rel-L2 {rel:.2e}, max|err|/rms {err.max() / rms:.2e}, "
          f"bf16-rounding exceptions {n_exc}")
    return rel, err.max() / rms, n_exc


def build(mx, w, set_idx=0):
    from mxfp4_expert_gb300 import synthetic
    layer = synthetic.build_layer(w, set_idx)
    x, bias = synthetic.inputs(w, set_idx)
    return layer, x, bias


@pytest.mark.parametrize("name,T,d,I,E,k,routing", [
    ("tiny", 1, 512, 128, 32, 4, "natural"),
    ("ragged", 5, 256, 64, 16, 3, "natural"),
    ("ragged", 17, 512, 96, 24, 5, "natural"),
    ("onehot", 3, 64, 32, 1, 1, "natural"),
    ("wide_k", 2, 128, 32, 40, 32, "natural"),
    ("mma_e600", 3, 256, 64, 600, 4, "natural"),   # E > 512: warp-MMA per-stage path
    ("three", 3, 256, 64, 16, 3, "natural"),
    ("four_small", 4, 512, 128, 32, 4, "natural"),
    # T >= 32: routed experts on the tcgen05 grouped GEMMs
    ("tc_tiny", 40, 512, 128, 32, 4, "natural"),
    ("tc_ragged", 33, 512, 96, 24, 5, "natural"),
    ("tc_wide_k", 32, 128, 32, 40, 32, "natural"),
    ("tc_many_rows", 300, 256, 64, 4, 2, "natural"),   # > 128 rows per expert: several token blocks
    # T >= 128: router, shared expert and combine on tcgen05 too; ragged T, E,
    # I and d against their 128-row blocks, K = d not a multiple of 64 (k3)
    ("tc_dense_ragged", 257, 384, 96, 136, 8, "natural"),
    ("tc_dense_k3", 200, 160, 224, 72, 3, "natural"),
])
def test_small_layers(mx, name, T, d, I, E, k, routing):
    w = wl.Workload(name, T=T, d=d, I=I, E=E, k=k, sets=1, routing=routing, seed=3)
    layer, x, bias = build(mx, w)
    out = run(mx, layer, x, bias, w.T, w.E, w.k)
    check_layer(w, 0, layer, x, bias, out)


def test_tc_items_beyond_table(mx):
    """tcgen05 path with more work items per CTA than its shared-memory item
    table holds (256): E=1024, k=32, ~130 rows per expert, so the down pass
    has about 49K items (d/128 row blocks x ceil(rows/64) token blocks per
    expert) and the items past the table are looked up on the fly."""
    w = wl.Workload("tc_items", T=4160, d=2048, I=32, E=1024, k=32, sets=1, routing="natural", seed=11)
    assert mx.moe_query_path(mx.moe_shape(w.d, w.I, w.E, w.k, True), w.T) == mx.MOE_PATH_PREFILL_TC
    layer, x, bias = build(mx, w)
    out = run(mx, layer, x, bias, w.T, w.E, w.k)
    counts = np.bincount(out[2].cpu().numpy().ravel(), minlength=w.E)
    items_down = int(sum((w.d // 128) * ((c + 63) // 64) for c in counts if c > 0))
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert items_down > 256 * sms, (items_down, sms)
    check_layer(w, 0, layer, x, bias, out, tokens=range(0, w.T, 347))


@pytest.mark.parametrize("T", [4, 40, 200])
def test_no_shared_expert(mx, T):
    """Without a shared expert: the single-launch kernel (T=4) and the
    tensor-core path (T=40, 200), where the dense stages stay on the warp-MMA
    kernels and the routed partials are combined by sorted slot."""
    from mxfp4_expert_gb300 import synthetic
    w = wl.Workload("noshared", T=T, d=256, I=64, E=16, k=2, sets=1, routing="natural", seed=5)
    full = synthetic.build_layer(w, 0)
    layer = mx.Layer(full.router_w, full.gate_up, full.struct.gate_up_desc, full.down,
                     full.struct.down_desc, top_k=w.k)
    x, _ = synthetic.inputs(w, 0)
    y, logits, idx, wts = run(mx, layer, x, None, w.T, w.E, w.k)
    gi = idx.cpu().numpy()
    experts = {e: omoe.Expert.from_fp32(*(t.cpu().numpy() for t in wl.gen_expert(w, 0, e, "cuda")))
               for e in set(gi.ravel().tolist())}
    ref = omoe.moe_layer(x.cpu(), full.router_w.cpu(), experts, None, w.k, idx=gi)
    yg = y.float().cpu().numpy()
    assert np.linalg.norm(yg - ref["y"]) / np.linalg.norm(ref["y"]) <= REL_L2


def test_ling_t1(mx):
    w = wl.get("ling_t1")
    for s in (0, 1):
        layer, x, bias = build(mx, w, s)
        out = run(mx, layer, x, bias, w.T, w.E, w.k)
        check_layer(w, s, layer, x, bias, out, strict=True)
        del layer
        torch.cuda.empty_cache()


def test_mtp_t4(mx):
    w = wl.get("mtp_t4")
    for s in (0, 5):
        layer, x, bias = build(mx, w, s)
        out = run(mx, layer, x, bias, w.T, w.E, w.k)
        D, sets = wl.mtp_expert_sets(w, s)
        assert len(set(out[2].cpu().numpy().ravel().tolist())) == D
        check_layer(w, s, layer, x, bias, out, strict=True)
        del layer
        torch.cuda.empty_cache()


@pytest.mark.parametrize("T", [5, 8, 16])
def test_ling_shape_small_t_tensor_core(mx, T):
    """Ling shapes at 5 <= T < 32 (the per-stage tcgen05 path with few tokens
    per expert), every token."""
    w = dataclasses.replace(wl.WORKLOADS["ling_t1"], name=f"ling_t{T}", T=T, sets=1)
    layer, x, bias = build(mx, w, 0)
    assert mx.moe_query_path(layer.shape, T) == mx.MOE_PATH_PREFILL_TC
    out = run(mx, layer, x, bias, w.T, w.E, w.k)
    check_layer(w, 0, layer, x, bias, out, strict=True)


def test_zipf_t64(mx):
    """T = 64 with Zipf(1.1) expert popularity: every token."""
    w = wl.get("zipf_t64")
    layer, x, bias = build(mx, w, 0)
    out = run(mx, layer, x, bias, w.T, w.E, w.k)
    D = len(set(out[2].cpu().numpy().ravel().tolist()))
    assert 100 <= D <= 220
    check_layer(w, 0, layer, x, bias, out, strict=True)


def covering_tokens(idx, E, at_least):
    """Tokens such that every expert in [0, E) is the choice of one of them
    (greedy set cover over the tokens' top-k sets), topped up with evenly
    spaced tokens to `at_least`; sorted."""
    T = idx.shape[0]
    sets = [set(r.tolist()) for r in idx]
    left, chosen = set(range(E)), set()
    while left:
        t = max(range(T), key=lambda i: (len(sets[i] & left), -i))
        if not sets[t] & left:
            break
        chosen.add(t)
        left -= sets[t]
    assert not left, f"experts never chosen: {sorted(left)[:8]}"
    for t in np.linspace(0, T - 1, at_least).astype(int):
        if len(chosen) >= at_least:
            break
        chosen.add(int(t))
    return sorted(chosen)


@pytest.mark.slow
def test_prefill_t4096(mx):
    """T = 4096: at least 256 tokens that between them choose all 512 experts,
    so every expert's work items on the grouped-GEMM path are checked."""
    w = wl.get("prefill_t4096")
    layer, x, bias = build(mx, w, 0)
    out = run(mx, layer, x, bias, w.T, w.E, w.k)
    toks = covering_tokens(out[2].cpu().numpy(), w.E, 256)
    assert len(toks) >= 256
    check_layer(w, 0, layer, x, bias, out, tokens=toks, strict=True)


def test_deterministic(mx):
    w = wl.get("mtp_t4")
    layer, x, bias = build(mx, w, 2)
    y1 = run(mx, layer, x, bias, w.T, w.E, w.k)[0].clone()
    y2 = run(mx, layer, x, bias, w.T, w.E, w.k)[0]
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_forward_rejects_bad_inputs(mx):
    w = wl.get("tiny")
    layer, x, bias = build(mx, w)
    bad = mx.Layer(layer.router_w, layer.gate_up, layer.struct.down_desc, layer.down, layer.struct.down_desc,
                   *layer.shared, top_k=w.k)
    with pytest.raises(mx.MoeError) as e:
        mx.moe_forward(bad, x)
    assert e.value.status == -3
    small = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(mx.MoeError) as e:
        mx.moe_forward(layer, x, workspace=small)
    assert e.value.status == -4
    with pytest.raises(mx.MoeError) as e:
        mx.moe_forward(layer, x, y=x)
    assert e.value.status == -1


def test_paths(mx):
    s = mx.moe_shape(2560, 768, 512, 8, 1)
    assert mx.moe_query_path(s, 1) == mx.MOE_PATH_DECODE_FUSED
    assert mx.moe_query_path(s, 4) == mx.MOE_PATH_DECODE_FUSED
    assert mx.moe_query_path(s, 5) == mx.MOE_PATH_PREFILL_TC
    assert mx.moe_query_path(s, 31) == mx.MOE_PATH_PREFILL_TC
    assert mx.moe_query_path(s, 32) == mx.MOE_PATH_PREFILL_TC
    # more than 512 experts do not fit the single-launch kernel: warp-MMA per-stage kernels
    assert mx.moe_query_path(mx.moe_shape(256, 64, 600, 4, 1), 3) == mx.MOE_PATH_DECODE_MMA
    assert mx.moe_query_path(s, 4096) == mx.MOE_PATH_PREFILL_TC
    assert mx.moe_stage_names(mx.MOE_PATH_DECODE_FUSED) == ["decode_fused"]
    assert len(mx.moe_stage_names(mx.MOE_PATH_DECODE_MMA)) == 8
    assert len(mx.moe_stage_names(mx.MOE_PATH_PREFILL_TC)) == 8


def test_fused_workspace_reuse_matches_fresh(mx):
    """The single-launch path keeps counters in the workspace between calls:
    a reused workspace must give bit-identical results to fresh ones."""
    from mxfp4_expert_gb300 import synthetic
    w = wl.get("mtp_t4")
    layers = [synthetic.build_layer(w, s) for s in (0, 1)]
    ins = [synthetic.inputs(w, s) for s in (0, 1)]
    fresh = [mx.moe_forward(layers[s], *ins[s]) for s in (0, 1)]
    ws = torch.zeros(layers[0].workspace_bytes(w.T), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for rep in range(5):
        s = rep % 2
        y = mx.moe_forward(layers[s], *ins[s], workspace=ws, dev_status=st)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), fresh[s].view(torch.int16)), rep
    assert int(st.item()) == 0


def test_bounded_wait_selftest(mx):
    """A wait on a flag that nothing sets gives up and reports MOE_DEV_TIMEOUT."""
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    mx.moe_selftest_bounded_wait(flag, 1, 2_000_000, st)
    torch.cuda.synchronize()
    assert int(st.item()) & mx.DEV_TIMEOUT
    st.zero_()
    flag.fill_(1)
    mx.moe_selftest_bounded_wait(flag, 1, 2_000_000, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
