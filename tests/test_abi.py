"""The C-ABI library loads and exports every function include/moe_mxfp4.h declares.

CPU only: no call here enqueues GPU work. Size/descriptor/status helpers are
host-only functions; argument checks return before any CUDA call.
"""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def mx():
    import __graft_entry__
    __graft_entry__.build()
    import mxfp4_expert_gb300 as mx
    return mx


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe_mxfp4.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)))


def test_header_symbols_exported(mx):
    names = declared_functions()
    assert len(names) >= 12
    out = subprocess.run(["nm", "-D", "--defined-only", mx.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (moe_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(mx.lib, n)


def test_status_strings_and_version(mx):
    assert mx.moe_status_string(0) == "ok"
    for code in range(-7, 0):
        assert mx.moe_status_string(code) != "unknown status"
    assert "sm_103a" in mx.moe_version()


def test_packed_bytes_and_descriptor(mx):
    assert mx.moe_packed_bytes(512, 1536, 2560, mx.MOE_LAYOUT_TILE16_GATEUP) == 512 * (1536 * 2560 // 2 + 1536 * 2560 // 32)
    assert mx.moe_packed_bytes(1, 2560, 768, mx.MOE_LAYOUT_TILE16) == 983040 + 61440
    assert mx.moe_packed_bytes(1, 24, 64, 1) == 0          # N not a multiple of 16
    assert mx.moe_packed_bytes(1, 32, 48, 1) == 0          # K not a multiple of 32
    assert mx.moe_packed_bytes(1, 32, 64, 7) == 0          # unknown layout
    d = mx.moe_describe_packed(3, 32, 64, 1)
    assert (d.magic, d.version, d.n_mat, d.N, d.K) == (0x3446584D, 2, 3, 32, 64)
    assert d.total_bytes == 3 * (32 * 64 // 2 + 32 * 64 // 32)
    with pytest.raises(mx.MoeError):
        mx.moe_describe_packed(1, 20, 64, 1)


def test_workspace_and_path_queries(mx):
    s = mx.moe_shape(2560, 768, 512, 8, 1)
    assert mx.moe_workspace_bytes(s, 1) > 0
    assert mx.moe_workspace_bytes(s, 64) > mx.moe_workspace_bytes(s, 1)
    # the path depends on the device; without one the query says so
    assert mx.moe_query_path(s, 1) in (mx.MOE_PATH_DECODE_MMA, mx.MOE_PATH_DECODE_FUSED, -7, -6)
    assert mx.moe_query_path(mx.moe_shape(2560, 768, 512, 600, 1), 1) == -2   # k > 32 / k > E
    assert mx.moe_query_path(mx.moe_shape(2560, 770, 512, 8, 1), 1) == -2     # I % 32
    assert mx.moe_workspace_bytes(mx.moe_shape(2560, 768, 2048, 8, 1), 1) == 0   # E > 1024


def test_argument_checks_return_before_cuda(mx):
    L = mx.lib
    assert L.moe_pack_mxfp4(None, 1, 16, 32, 1, None, 0, None, None, None) == -1
    assert L.moe_route_topk(None, 1, 8, 2, None, 0, None, None, None) == -1
    assert L.moe_forward(None, None, 1, None, None, 0, None, None, None, None, 0, None, None, 0, None) == -1
    assert L.moe_sort_by_expert(None, 1, 1, 1, None, None, None, None, None, None, None, 0, None, None) == -1
    assert L.moe_unpack_mxfp4(None, None, None, None, None) == -1
    # a descriptor with the wrong magic is refused before any device work
    bad = mx.moe_packed_desc(0xDEAD, 1, 1, 1, 16, 32, 272, 272)
    p = ctypes.c_void_p(16)
    assert L.moe_unpack_mxfp4(p, ctypes.byref(bad), p, p, None) == -3


def test_binding_refuses_missing_library(tmp_path):
    code = ("import sys; sys.path.insert(0, %r); import mxfp4_expert_gb300 as m" % ROOT)
    env = dict(os.environ)
    # a copy of the package without the library must fail at import, loudly
    import shutil
    pkg = tmp_path / "mxfp4_expert_gb300"
    shutil.copytree(os.path.join(ROOT, "mxfp4_expert_gb300"), pkg,
                    ignore=shutil.ignore_patterns("*.so", "_build", "__pycache__"))
    shutil.copytree(os.path.join(ROOT, "workloads"), tmp_path / "workloads")
    r = subprocess.run(["python", "-c", code.replace(repr(ROOT), repr(str(tmp_path)))],
                       capture_output=True, text=True, env=env)
    assert r.returncode != 0 and "libmoe_mxfp4.so is missing" in r.stderr
