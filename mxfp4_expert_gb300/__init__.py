"""Python binding of libmoe_mxfp4 — the GB300 (sm_103a) MXFP4 mixture-of-experts layer.

The functions here carry the C-ABI names (see include/moe_mxfp4.h) and only
marshal arguments: every step of the layer runs in the library's CUDA
kernels. PyTorch supplies device memory and streams. There is no CPU or
PyTorch fallback: importing this package fails if the library has not been
built, and every call raises ``MoeError`` on a non-zero status.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "MoeError", "LIB_PATH", "lib", "MOE_LAYOUT_TILE16", "MOE_LAYOUT_TILE16_GATEUP",
    "MOE_PATH_DECODE_MMA", "MOE_PATH_DECODE_FUSED", "MOE_PATH_PREFILL_TC", "DEV_NONFINITE_INPUT", "DEV_SCALE_RANGE", "DEV_INDEX_OOB", "DEV_TIMEOUT",
    "moe_packed_desc", "moe_shape", "moe_layer", "Layer",
    "moe_packed_bytes", "moe_describe_packed", "moe_pack_mxfp4", "moe_unpack_mxfp4",
    "moe_route_topk", "moe_sort_workspace_bytes", "moe_sort_by_expert",
    "moe_workspace_bytes", "moe_query_path", "moe_stage_names", "moe_forward", "moe_forward_profiled", "moe_forward_w4a8", "moe_quant_mxfp8", "moe_lmhead_pack_fp8", "moe_lmhead_fp8", "moe_forward_static_scratch", "STATIC_SCRATCH_BYTES", "moe_selftest_bounded_wait", "moe_status_string", "moe_version",
]

# The in-tree build, and only it: there is no way to point the binding at
# another library.
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe_mxfp4.so")
# Version string the library must report (moe_version); anything else is refused.
EXPECTED_VERSION = "moe_mxfp4 1.2 sm_103a"

MOE_LAYOUT_TILE16 = 1
MOE_LAYOUT_TILE16_GATEUP = 2
MOE_PATH_DECODE_MMA = 1
MOE_PATH_DECODE_FUSED = 2
MOE_PATH_PREFILL_TC = 3
DEV_NONFINITE_INPUT, DEV_SCALE_RANGE, DEV_INDEX_OOB, DEV_TIMEOUT = 1, 2, 4, 8
STATIC_SCRATCH_BYTES = 4 * 1024 * 1024


class MoeError(RuntimeError):
    def __init__(self, what: str, status: int):
        super().__init__(f"{what}: {moe_status_string(status)} (status {status})")
        self.status = status


class moe_packed_desc(ctypes.Structure):
    _fields_ = [("magic", ctypes.c_uint32), ("version", ctypes.c_uint32), ("layout", ctypes.c_int32),
                ("n_mat", ctypes.c_int32), ("N", ctypes.c_int32), ("K", ctypes.c_int32),
                ("bytes_per_mat", ctypes.c_uint64), ("total_bytes", ctypes.c_uint64)]


class moe_shape(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int32), ("d_ff", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("has_shared", ctypes.c_int32)]


class moe_layer(ctypes.Structure):
    _fields_ = [("shape", moe_shape), ("router_w", ctypes.c_void_p),
                ("gate_up", ctypes.c_void_p), ("gate_up_desc", moe_packed_desc),
                ("down", ctypes.c_void_p), ("down_desc", moe_packed_desc),
                ("shared_gate", ctypes.c_void_p), ("shared_up", ctypes.c_void_p),
                ("shared_down", ctypes.c_void_p)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing. Build it with `python -c \"import __graft_entry__ as g; g.build()\"` "
            "(nvcc, sm_103a). This package has no CPU or PyTorch fallback.")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    sig = {
        "moe_packed_bytes": (sz, [i32, i32, i32, i32]),
        "moe_describe_packed": (i32, [i32, i32, i32, i32, ctypes.POINTER(moe_packed_desc)]),
        "moe_pack_mxfp4": (i32, [vp, i32, i32, i32, i32, vp, sz, ctypes.POINTER(moe_packed_desc), vp, vp]),
        "moe_unpack_mxfp4": (i32, [vp, ctypes.POINTER(moe_packed_desc), vp, vp, vp]),
        "moe_route_topk": (i32, [vp, i32, i32, i32, vp, i32, vp, vp, vp]),
        "moe_sort_workspace_bytes": (sz, [i32, i32, i32]),
        "moe_sort_by_expert": (i32, [vp, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp]),
        "moe_workspace_bytes": (sz, [ctypes.POINTER(moe_shape), i32]),
        "moe_query_path": (i32, [ctypes.POINTER(moe_shape), i32]),
        "moe_forward": (i32, [ctypes.POINTER(moe_layer), vp, i32, vp, vp, i32, vp, vp, vp, vp, sz, vp, vp]),
        "moe_lmhead_pack_fp8": (i32, [vp, i32, i32, vp, vp, vp]),
        "moe_lmhead_fp8": (i32, [vp, vp, i32, i32, vp, i32, vp, vp]),
        "moe_quant_mxfp8": (i32, [vp, i32, i32, i32, vp, vp, vp]),
        "moe_forward_w4a8": (i32, [ctypes.POINTER(moe_layer), vp, i32, vp, vp, i32, vp, vp, vp, vp, sz, vp, vp]),
        "moe_forward_profiled": (i32, [ctypes.POINTER(moe_layer), vp, i32, vp, vp, i32, vp, vp, vp, vp, sz, vp,
                                         ctypes.POINTER(ctypes.c_void_p), i32, vp]),
        "moe_forward_static_scratch": (i32, [ctypes.POINTER(moe_layer), vp, i32, vp, vp, i32, vp, vp, vp, vp, vp]),
        "moe_stage_names": (ctypes.c_char_p, [i32]),
        "moe_selftest_bounded_wait": (i32, [vp, ctypes.c_uint32, ctypes.c_longlong, vp, vp]),
        "moe_status_string": (ctypes.c_char_p, [i32]),
        "moe_version": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype, f.argtypes = res, args
    got = L.moe_version().decode()
    if got != EXPECTED_VERSION:
        raise ImportError(f"{LIB_PATH} reports version {got!r}, this binding needs {EXPECTED_VERSION!r}; rebuild it")
    return L


lib = _load()


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _s(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(status: int, what: str):
    if status != 0:
        raise MoeError(what, status)


def _cuda(t, dtype, name):
    if not (isinstance(t, torch.Tensor) and t.is_cuda):
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def moe_selftest_bounded_wait(flag: torch.Tensor, want: int, budget_cycles: int,
                              dev_status: torch.Tensor, stream=None):
    """Run the kernels' bounded wait on flag (uint32 as int32 tensor) == want."""
    _check(lib.moe_selftest_bounded_wait(_p(flag), want, budget_cycles, _p(dev_status), _s(stream)),
           "moe_selftest_bounded_wait")


def moe_status_string(status: int) -> str:
    return lib.moe_status_string(status).decode()


def moe_version() -> str:
    return lib.moe_version().decode()


def moe_packed_bytes(n_mat: int, N: int, K: int, layout: int) -> int:
    return int(lib.moe_packed_bytes(n_mat, N, K, layout))


def moe_describe_packed(n_mat: int, N: int, K: int, layout: int) -> moe_packed_desc:
    d = moe_packed_desc()
    _check(lib.moe_describe_packed(n_mat, N, K, layout, ctypes.byref(d)), "moe_describe_packed")
    return d


def moe_pack_mxfp4(w: torch.Tensor, layout: int, out: torch.Tensor | None = None,
                   dev_status: torch.Tensor | None = None, stream=None):
    """fp32 [n_mat, N, K] (or [N, K]) -> (packed uint8 tensor, moe_packed_desc)."""
    _cuda(w, torch.float32, "w")
    n_mat, N, K = (1, *w.shape) if w.dim() == 2 else tuple(w.shape)
    nbytes = moe_packed_bytes(n_mat, N, K, layout)
    if nbytes == 0:
        raise MoeError("moe_pack_mxfp4", -2)
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=w.device)
    desc = moe_packed_desc()
    _check(lib.moe_pack_mxfp4(_p(w), n_mat, N, K, layout, _p(out), out.numel(), ctypes.byref(desc),
                              _p(dev_status), _s(stream)), "moe_pack_mxfp4")
    return out, desc


def moe_unpack_mxfp4(packed: torch.Tensor, desc: moe_packed_desc, stream=None):
    """Packed buffer -> canonical (codes [n_mat, N, K/2], scales [n_mat, N, K/32]) uint8."""
    codes = torch.empty((desc.n_mat, desc.N, desc.K // 2), dtype=torch.uint8, device=packed.device)
    scales = torch.empty((desc.n_mat, desc.N, desc.K // 32), dtype=torch.uint8, device=packed.device)
    _check(lib.moe_unpack_mxfp4(_p(packed), ctypes.byref(desc), _p(codes), _p(scales), _s(stream)),
           "moe_unpack_mxfp4")
    return codes, scales


def moe_route_topk(logits: torch.Tensor, k: int, bias: torch.Tensor | None = None,
                   idx: torch.Tensor | None = None, w: torch.Tensor | None = None, stream=None):
    """fp32 logits [T, E] -> (idx int32 [T, k], w fp32 [T, k]); bias [E] or [T, E]."""
    _cuda(logits, torch.float32, "logits")
    T, E = logits.shape
    stride = 0
    if bias is not None:
        _cuda(bias, torch.float32, "bias")
        stride = 0 if bias.dim() == 1 else bias.shape[1]
    idx = torch.empty((T, k), dtype=torch.int32, device=logits.device) if idx is None else idx
    w = torch.empty((T, k), dtype=torch.float32, device=logits.device) if w is None else w
    _check(lib.moe_route_topk(_p(logits), T, E, k, _p(bias), stride, _p(idx), _p(w), _s(stream)),
           "moe_route_topk")
    return idx, w


def moe_sort_workspace_bytes(T: int, k: int, E: int) -> int:
    return int(lib.moe_sort_workspace_bytes(T, k, E))


def moe_sort_by_expert(idx: torch.Tensor, E: int, dev_status: torch.Tensor | None = None, stream=None):
    """int32 idx [T, k] -> dict(counts, offsets, perm, inv, active, n_active) device tensors."""
    _cuda(idx, torch.int32, "idx")
    T, k = idx.shape
    dev = idx.device
    out = {"counts": torch.empty(E, dtype=torch.int32, device=dev),
           "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
           "perm": torch.empty(T * k, dtype=torch.int32, device=dev),
           "inv": torch.empty(T * k, dtype=torch.int32, device=dev),
           "active": torch.empty(E, dtype=torch.int32, device=dev),
           "n_active": torch.empty(1, dtype=torch.int32, device=dev)}
    nws = moe_sort_workspace_bytes(T, k, E)
    ws = torch.empty(max(nws, 256), dtype=torch.uint8, device=dev)
    _check(lib.moe_sort_by_expert(_p(idx), T, k, E, _p(out["counts"]), _p(out["offsets"]), _p(out["perm"]),
                                  _p(out["inv"]), _p(out["active"]), _p(out["n_active"]), _p(ws), ws.numel(),
                                  _p(dev_status), _s(stream)), "moe_sort_by_expert")
    return out


def _shape(d, I, E, k, has_shared) -> moe_shape:
    return moe_shape(d, I, E, k, 1 if has_shared else 0)


def moe_workspace_bytes(shape: moe_shape, T: int) -> int:
    return int(lib.moe_workspace_bytes(ctypes.byref(shape), T))


def moe_query_path(shape: moe_shape, T: int) -> int:
    return int(lib.moe_query_path(ctypes.byref(shape), T))


def moe_stage_names(path: int) -> list[str]:
    r = lib.moe_stage_names(path)
    return [] if r is None else r.decode().split(",")


class Layer:
    """Device weights of one layer plus the moe_layer struct the C ABI takes.

    router_w bf16 [E, d]; gate_up packed (layout TILE16_GATEUP, n_mat=E, N=2I,
    K=d); down packed (layout TILE16, n_mat=E, N=d, K=I); shared_* bf16 or None.
    """

    def __init__(self, router_w, gate_up, gate_up_desc, down, down_desc,
                 shared_gate=None, shared_up=None, shared_down=None, top_k=8):
        E, d = router_w.shape
        I = gate_up_desc.N // 2
        self.router_w, self.gate_up, self.down = router_w, gate_up, down
        self.shared = (shared_gate, shared_up, shared_down)
        has_shared = shared_gate is not None
        self.shape = _shape(d, I, E, top_k, has_shared)
        self.struct = moe_layer(self.shape, router_w.data_ptr(), gate_up.data_ptr(), gate_up_desc,
                                down.data_ptr(), down_desc,
                                shared_gate.data_ptr() if has_shared else None,
                                shared_up.data_ptr() if has_shared else None,
                                shared_down.data_ptr() if has_shared else None)

    @classmethod
    def from_fp32(cls, router_w, gate_up_f32, down_f32, shared=None, top_k=8, stream=None):
        """Pack fp32 expert weights (gate_up [E, 2I, d], down [E, d, I]) with moe_pack_mxfp4."""
        gu, gud = moe_pack_mxfp4(gate_up_f32, MOE_LAYOUT_TILE16_GATEUP, stream=stream)
        dn, dnd = moe_pack_mxfp4(down_f32, MOE_LAYOUT_TILE16, stream=stream)
        sg, su, sd = shared if shared is not None else (None, None, None)
        return cls(router_w, gu, gud, dn, dnd, sg, su, sd, top_k=top_k)

    @property
    def d(self):
        return self.shape.d_model

    def workspace_bytes(self, T: int) -> int:
        return moe_workspace_bytes(self.shape, T)


def _forward_args(layer: Layer, x, bias, y, logits_out, idx_out, w_out, dev_status):
    """Checks shared by the forward calls; returns (T, bias row stride).

    The C library can only check pointers and sizes it is given; these checks
    make sure every tensor is large enough for what the kernels write or read,
    and that all of them live on the current device."""
    _cuda(x, torch.bfloat16, "x")
    _cuda(y, torch.bfloat16, "y")
    if x.dim() != 2 or x.shape[1] != layer.d:
        raise ValueError(f"x must be [T, {layer.d}], got {tuple(x.shape)}")
    if y.shape != x.shape:
        raise ValueError(f"y must have x's shape {tuple(x.shape)}, got {tuple(y.shape)}")
    T, E, k = x.shape[0], layer.shape.n_experts, layer.shape.top_k
    dev = torch.cuda.current_device()
    stride = 0
    if bias is not None:
        _cuda(bias, torch.float32, "bias")
        if bias.dim() == 1:
            if bias.numel() != E:
                raise ValueError(f"bias must have {E} entries")
        elif bias.dim() == 2 and bias.shape[0] >= T and bias.shape[1] == E:
            stride = E
        else:
            raise ValueError(f"bias must be [{E}] or [T, {E}], got {tuple(bias.shape)}")
    for name, t, dtype, n in (("logits_out", logits_out, torch.float32, T * E),
                              ("idx_out", idx_out, torch.int32, T * k),
                              ("w_out", w_out, torch.float32, T * k),
                              ("dev_status", dev_status, torch.int32, 1)):
        if t is not None:
            _cuda(t, dtype, name)
            if t.numel() < n:
                raise ValueError(f"{name} needs at least {n} elements, got {t.numel()}")
    for name, t in (("x", x), ("y", y), ("bias", bias), ("logits_out", logits_out), ("idx_out", idx_out),
                    ("w_out", w_out), ("dev_status", dev_status)):
        if t is not None and t.device.index != dev:
            raise ValueError(f"{name} is on cuda:{t.device.index}, the current device is cuda:{dev}")
    return T, stride


def moe_forward(layer: Layer, x: torch.Tensor, bias: torch.Tensor | None = None,
                y: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                logits_out: torch.Tensor | None = None, idx_out: torch.Tensor | None = None,
                w_out: torch.Tensor | None = None, dev_status: torch.Tensor | None = None,
                stream=None):
    """y = layer(x) for bf16 x [T, d]; returns y (bf16 [T, d]).

    workspace: uint8 device tensor of layer.workspace_bytes(T) bytes, zero-filled
    before its first use (it carries synchronisation counters between calls);
    allocated with zeros when omitted.
    """
    return _forward(layer, x, bias, y, workspace, logits_out, idx_out, w_out, dev_status, None, stream)


def moe_forward_w4a8(layer: Layer, x: torch.Tensor, bias: torch.Tensor | None = None,
                     y: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                     logits_out: torch.Tensor | None = None, idx_out: torch.Tensor | None = None,
                     w_out: torch.Tensor | None = None, dev_status: torch.Tensor | None = None,
                     stream=None):
    """The layer with MXFP8 activations before each routed-expert GEMM (W4A8),
    on the block-scaled tcgen05 path for any T; otherwise as moe_forward."""
    return _forward(layer, x, bias, y, workspace, logits_out, idx_out, w_out, dev_status, None, stream,
                    entry="moe_forward_w4a8")


def moe_quant_mxfp8(src: torch.Tensor, stream=None):
    """bf16 or fp32 [rows, K] -> (E4M3 codes uint8 [rows, K], E8M0 scales uint8 [rows, K/32])."""
    if src.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("src must be bf16 or fp32")
    _cuda(src, src.dtype, "src")
    rows, K = src.shape
    codes = torch.empty((rows, K), dtype=torch.uint8, device=src.device)
    scales = torch.empty((rows, K // 32), dtype=torch.uint8, device=src.device)
    _check(lib.moe_quant_mxfp8(_p(src), 1 if src.dtype == torch.bfloat16 else 0, rows, K, _p(codes), _p(scales),
                               _s(stream)), "moe_quant_mxfp8")
    return codes, scales


def moe_lmhead_pack_fp8(w: torch.Tensor, stream=None):
    """bf16 LM head [V, d] -> (E4M3 codes uint8 [V, d], fp32 row scales [V])."""
    _cuda(w, torch.bfloat16, "w")
    V, d = w.shape
    codes = torch.empty((V, d), dtype=torch.uint8, device=w.device)
    scales = torch.empty(V, dtype=torch.float32, device=w.device)
    _check(lib.moe_lmhead_pack_fp8(_p(w), V, d, _p(codes), _p(scales), _s(stream)), "moe_lmhead_pack_fp8")
    return codes, scales


def moe_lmhead_fp8(codes: torch.Tensor, scales: torch.Tensor, x: torch.Tensor, logits: torch.Tensor | None = None,
                   stream=None):
    """fp32 logits [T, V] of bf16 x [T, d] against the FP8 head (codes, scales)."""
    _cuda(codes, torch.uint8, "codes")
    _cuda(scales, torch.float32, "scales")
    _cuda(x, torch.bfloat16, "x")
    V, d = codes.shape
    if x.dim() != 2 or x.shape[1] != d or scales.numel() != V:
        raise ValueError("x must be [T, d] and scales [V] for codes [V, d]")
    T = x.shape[0]
    if logits is None:
        logits = torch.empty((T, V), dtype=torch.float32, device=x.device)
    _cuda(logits, torch.float32, "logits")
    if logits.numel() < T * V:
        raise ValueError("logits needs T * V elements")
    _check(lib.moe_lmhead_fp8(_p(codes), _p(scales), V, d, _p(x), T, _p(logits), _s(stream)), "moe_lmhead_fp8")
    return logits


def moe_forward_profiled(layer: Layer, x: torch.Tensor, stage_events, bias: torch.Tensor | None = None,
                         y: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                         logits_out: torch.Tensor | None = None, idx_out: torch.Tensor | None = None,
                         w_out: torch.Tensor | None = None, dev_status: torch.Tensor | None = None,
                         stream=None):
    """moe_forward that also records `stage_events` (torch.cuda.Event with
    enable_timing=True) at its stage boundaries; see moe_stage_names."""
    return _forward(layer, x, bias, y, workspace, logits_out, idx_out, w_out, dev_status, list(stage_events),
                    stream)


def _forward(layer, x, bias, y, workspace, logits_out, idx_out, w_out, dev_status, stage_events, stream,
             entry="moe_forward"):
    if y is None:
        _cuda(x, torch.bfloat16, "x")
        y = torch.empty_like(x)
    T, stride = _forward_args(layer, x, bias, y, logits_out, idx_out, w_out, dev_status)
    if workspace is None:
        workspace = torch.zeros(layer.workspace_bytes(T), dtype=torch.uint8, device=x.device)
    _cuda(workspace, torch.uint8, "workspace")
    args = (ctypes.byref(layer.struct), _p(x), T, _p(y), _p(bias), stride, _p(logits_out), _p(idx_out), _p(w_out),
            _p(workspace), workspace.numel(), _p(dev_status))
    if stage_events is None:
        _check(getattr(lib, entry)(*args, _s(stream)), entry)
    else:
        n_ev = len(stage_events)
        ev_arr = (ctypes.c_void_p * n_ev)(*[e.cuda_event for e in stage_events])
        _check(lib.moe_forward_profiled(*args, ev_arr, n_ev, _s(stream)), "moe_forward_profiled")
    return y


def moe_forward_static_scratch(layer: Layer, x: torch.Tensor, y: torch.Tensor, bias: torch.Tensor | None = None,
                               logits_out: torch.Tensor | None = None, idx_out: torch.Tensor | None = None,
                               w_out: torch.Tensor | None = None, dev_status: torch.Tensor | None = None,
                               stream=None):
    """y = layer(x) without a workspace and without allocating: the library's
    fixed device scratch array (STATIC_SCRATCH_BYTES per device) stands in
    for it. y (bf16 [T, d]) is the caller's. Calls on one device share that
    array, so calls that may overlap in time must be ordered by the caller;
    the first call on a device should come before any stream capture.
    Every tensor is checked (shape, size, dtype, current device) before the
    call, so a wrong buffer raises instead of letting a kernel run past it.
    """
    T, stride = _forward_args(layer, x, bias, y, logits_out, idx_out, w_out, dev_status)
    _check(lib.moe_forward_static_scratch(ctypes.byref(layer.struct), _p(x), T, _p(y), _p(bias), stride,
                                          _p(logits_out), _p(idx_out), _p(w_out), _p(dev_status), _s(stream)),
           "moe_forward_static_scratch")
    return y
