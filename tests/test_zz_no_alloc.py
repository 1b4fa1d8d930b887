"""moe_forward_static_scratch (no workspace, no allocation) against moe_forward.

The file name sorts last so that pytest runs it after every other test; it
must also pass on its own in a fresh process, where its first call is the one
that looks up the library's scratch array.

Two calls in a row through the static-scratch entry point, on different
inputs, each compared with moe_forward (own zero-filled workspace) on the
same inputs: indices bit-exact, and y within the layer tests' tolerance
(relative L2 <= 5e-3, max |err| <= 2e-2 * rms of moe_forward's y).
"""
import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu

REL_L2 = 5e-3
MAX_ABS = 2e-2


@pytest.fixture(scope="module")
def mx():
    import mxfp4_expert_gb300 as mx
    return mx


def _outputs(T, E, k):
    return (torch.empty((T, E), dtype=torch.float32, device="cuda"),
            torch.empty((T, k), dtype=torch.int32, device="cuda"),
            torch.empty((T, k), dtype=torch.float32, device="cuda"),
            torch.zeros(1, dtype=torch.int32, device="cuda"))


def _compare(mx, layer, x, bias, w):
    T, E, k = x.shape[0], w.E, w.k
    l_r, i_r, w_r, s_r = _outputs(T, E, k)
    y_r = mx.moe_forward(layer, x, bias, logits_out=l_r, idx_out=i_r, w_out=w_r, dev_status=s_r)
    l_s, i_s, w_s, s_s = _outputs(T, E, k)
    y_s = torch.empty_like(x)
    mx.moe_forward_static_scratch(layer, x, y_s, bias, logits_out=l_s, idx_out=i_s, w_out=w_s, dev_status=s_s)
    torch.cuda.synchronize()
    assert int(s_r.item()) == 0 and int(s_s.item()) == 0
    assert torch.equal(i_s, i_r)
    assert torch.allclose(w_s, w_r, rtol=0, atol=2e-6)
    yr = y_r.float().cpu().numpy().astype(np.float64)
    ys = y_s.float().cpu().numpy().astype(np.float64)
    rel = np.linalg.norm(ys - yr) / np.linalg.norm(yr)
    rms = np.sqrt(np.mean(yr ** 2))
    assert rel <= REL_L2, rel
    assert np.max(np.abs(ys - yr)) <= MAX_ABS * rms


def _x(w, set_idx, T):
    g = torch.Generator(device="cpu").manual_seed(9000 + 31 * set_idx + T)
    return (torch.randn((T, w.d), generator=g) * 0.5).to(torch.bfloat16).cuda()


@pytest.mark.parametrize("name,T", [("tiny", None), ("ling_t1", 1), ("ling_t1", 4), ("ling_t1", 8)])
def test_static_scratch_matches_moe_forward_twice(mx, name, T):
    from mxfp4_expert_gb300 import synthetic
    w = wl.WORKLOADS[name]
    layer = synthetic.build_layer(w, 0)
    T = w.T if T is None else T
    assert mx.moe_workspace_bytes(layer.shape, T) <= mx.STATIC_SCRATCH_BYTES
    for call in range(2):
        _compare(mx, layer, _x(w, call, T), None, w)


def test_static_scratch_ling_limit(mx):
    """At the Ling shape the 4 MiB array holds the workspace of up to 26
    tokens: T = 26 runs (and matches moe_forward), T = 27 is refused with
    MOE_ERR_WORKSPACE_TOO_SMALL before anything is enqueued."""
    from mxfp4_expert_gb300 import synthetic
    w = wl.WORKLOADS["ling_t1"]
    layer = synthetic.build_layer(w, 0)
    assert mx.moe_workspace_bytes(layer.shape, 26) <= mx.STATIC_SCRATCH_BYTES
    assert mx.moe_workspace_bytes(layer.shape, 27) > mx.STATIC_SCRATCH_BYTES
    _compare(mx, layer, _x(w, 0, 26), None, w)
    x = _x(w, 1, 27)
    y = torch.full_like(x, 7.0)
    with pytest.raises(mx.MoeError) as ei:
        mx.moe_forward_static_scratch(layer, x, y)
    assert ei.value.status == -4
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())


def test_static_scratch_allocates_nothing(mx):
    """A warmed-up call changes neither the device's free memory nor the
    caching allocator's reserved bytes."""
    from mxfp4_expert_gb300 import synthetic
    w = wl.WORKLOADS["ling_t1"]
    layer = synthetic.build_layer(w, 0)
    x = _x(w, 2, 4)
    y = torch.empty_like(x)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    mx.moe_forward_static_scratch(layer, x, y, dev_status=st)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    res0 = torch.cuda.memory_reserved()
    for _ in range(3):
        mx.moe_forward_static_scratch(layer, x, y, dev_status=st)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0 and torch.cuda.memory_reserved() == res0
    assert int(st.item()) == 0


def test_static_scratch_after_a_timed_out_wait(mx):
    """Each call clears the counters it needs, so it does not depend on how an
    earlier kernel ended: after a bounded wait that gave up (a flag nothing
    sets), the next call still matches moe_forward."""
    from mxfp4_expert_gb300 import synthetic
    w = wl.WORKLOADS["ling_t1"]
    layer = synthetic.build_layer(w, 0)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    mx.moe_selftest_bounded_wait(flag, 1, 2_000_000, st)
    torch.cuda.synchronize()
    assert int(st.item()) & mx.DEV_TIMEOUT
    _compare(mx, layer, _x(w, 3, 1), None, w)


def test_static_scratch_checks_buffers(mx):
    """Buffers too small for what the kernels write, or of the wrong width, are
    refused by the binding before the library is called."""
    from mxfp4_expert_gb300 import synthetic
    w = wl.WORKLOADS["tiny"]
    layer = synthetic.build_layer(w, 0)
    x = _x(w, 0, 2)
    with pytest.raises(ValueError):
        mx.moe_forward_static_scratch(layer, x, torch.empty((1, w.d), dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(ValueError):
        mx.moe_forward_static_scratch(layer, x[:, :256].contiguous(), torch.empty((2, 256), dtype=torch.bfloat16,
                                                                                 device="cuda"))
    with pytest.raises(ValueError):
        mx.moe_forward_static_scratch(layer, x, torch.empty_like(x),
                                      logits_out=torch.empty(w.E, dtype=torch.float32, device="cuda"))
    with pytest.raises(ValueError):
        mx.moe_forward_static_scratch(layer, x, torch.empty_like(x),
                                      idx_out=torch.empty(w.k, dtype=torch.int32, device="cuda"))


def test_static_scratch_rejects_too_large(mx):
    from mxfp4_expert_gb300 import synthetic
    w = wl.WORKLOADS["tiny"]
    layer = synthetic.build_layer(w, 0)
    T = 1
    while mx.moe_workspace_bytes(layer.shape, T) <= mx.STATIC_SCRATCH_BYTES:
        T *= 2
    x = _x(w, 0, T)
    y = torch.empty_like(x)
    with pytest.raises(mx.MoeError) as ei:
        mx.moe_forward_static_scratch(layer, x, y)
    assert ei.value.status == -4  # MOE_ERR_WORKSPACE_TOO_SMALL
