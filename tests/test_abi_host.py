"""The C-ABI library on the host (no GPU): it loads, exports every function
include/lily_moe.h declares, sizes workspaces, and rejects bad arguments
before launching anything."""
import ctypes
import re
from pathlib import Path

import pytest

import w4_grouped_gemm_gb300 as lily
from w4_grouped_gemm_gb300 import _lib

HEADER = Path(__file__).resolve().parent.parent / "include" / "lily_moe.h"


@pytest.fixture(scope="module")
def L():
    from w4_grouped_gemm_gb300 import build
    build.build()
    return lily.lib()


def _declared_functions():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lily_moe_\w+)\s*\(", text)))


def test_header_functions_exported(L):
    names = _declared_functions()
    assert len(names) >= 16
    for n in names:
        assert hasattr(L, n), f"{n} declared in lily_moe.h but not exported"
    assert sorted(_lib.EXPORTS) == names


def test_version_and_strerror(L):
    assert "sm_103a" in lily.lily_moe_version()
    for code in range(0, -8, -1):
        assert lily.strerror(code) != "unknown error"


def test_check_dims():
    ok = lily.make_dims(512, 2048, 256, 8, 512, 128)
    assert lily.lily_moe_check_dims(ok) == 0
    bad = [
        lily.make_dims(0, 2048, 256, 8, 512, 128),
        lily.make_dims(512, 2000, 256, 8, 512, 128),
        lily.make_dims(512, 2048, 300, 8, 512, 128),
        lily.make_dims(512, 2048, 256, 9, 512, 128),
        lily.make_dims(512, 2048, 4, 8, 512, 128),
        lily.make_dims(512, 2048, 256, 8, 500, 128),
        lily.make_dims(512, 2048, 256, 8, 512, 48),
        lily.make_dims(512, 2048, 256, 8, 512, 256),
        lily.make_dims(512, 2048, 256, 8, 512, 128, group=32),
        lily.make_dims(20000, 2048, 256, 8, 512, 128),
        lily.make_dims(512, 2048, 256, 8, 512, 128, out_dtype=7),
    ]
    for d in bad:
        assert lily.lily_moe_check_dims(d) < 0
        assert lily.lily_moe_workspace_bytes(d) == 0


def test_block_map_cap_and_workspace():
    d = lily.make_dims(2048, 2048, 256, 8, 512, 128)
    assert lily.lily_moe_block_map_cap(d) == 16384 // 128 + 256
    d = lily.make_dims(1, 2048, 256, 8, 512, 32)
    assert lily.lily_moe_block_map_cap(d) == 1 + 8
    ws = lily.lily_moe_workspace_bytes(lily.make_dims(2048, 2048, 256, 8, 512, 128))
    # at least H (P+T rows of F bf16) and the fp32 accumulator
    assert ws >= (16384 + 2048) * 512 * 2 + 2048 * 2048 * 4
    assert lily.lily_moe_stack_workspace_bytes(lily.make_dims(2048, 2048, 256, 8, 512, 128)) > ws


def _call_forward(L, dims, x=16, w=True, r=True, y=16, ws=16, ws_bytes=1 << 40):
    wt = _lib.Weights(*([256] * 11)) if w else None
    rt = _lib.Routing(*([256] * 9)) if r else None
    return L.lily_moe_forward(ctypes.byref(dims), x, ctypes.byref(wt) if wt else None,
                              ctypes.byref(rt) if rt else None, y, ws, ws_bytes, None)


def test_argument_errors_launch_nothing(L):
    """Each bad argument returns its code before any CUDA call (no GPU here)."""
    d = lily.make_dims(64, 512, 32, 4, 128, 32)
    assert _call_forward(L, d, x=None) == lily.LILY_ERR_INVALID_ARG
    assert _call_forward(L, d, y=None) == lily.LILY_ERR_INVALID_ARG
    assert _call_forward(L, d, w=False) == lily.LILY_ERR_INVALID_ARG
    assert _call_forward(L, d, r=False) == lily.LILY_ERR_INVALID_ARG
    assert _call_forward(L, d, ws=None) == lily.LILY_ERR_INVALID_ARG
    assert _call_forward(L, d, x=24) == lily.LILY_ERR_MISALIGNED
    assert _call_forward(L, d, ws=8) == lily.LILY_ERR_MISALIGNED
    assert _call_forward(L, d, ws_bytes=100) == lily.LILY_ERR_WORKSPACE_TOO_SMALL
    bad = lily.make_dims(64, 500, 32, 4, 128, 32)
    assert _call_forward(L, bad) == lily.LILY_ERR_UNSUPPORTED_SHAPE
    wt = _lib.Weights(*([256] * 11))
    wt.gate_q = 260
    rt = _lib.Routing(*([256] * 9))
    assert L.lily_moe_forward(ctypes.byref(d), 16, ctypes.byref(wt), ctypes.byref(rt), 16, 16,
                              1 << 40, None) == lily.LILY_ERR_MISALIGNED
    # decode refuses T > 8 before touching the device
    d9 = lily.make_dims(9, 512, 32, 4, 128, 32)
    wt = _lib.Weights(*([256] * 11))
    rc = L.lily_moe_decode(ctypes.byref(d9), 16, ctypes.byref(wt), ctypes.byref(rt), 16, 16, 1 << 40,
                           None)
    assert rc in (lily.LILY_ERR_UNSUPPORTED_SHAPE, lily.LILY_ERR_CUDA, lily.LILY_ERR_ARCH)
    assert L.lily_moe_status(None, None) == lily.LILY_ERR_INVALID_ARG


def test_no_gpu_reports_cuda_or_arch_error(L):
    """With valid arguments but no device, the call fails cleanly."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    d = lily.make_dims(64, 512, 32, 4, 128, 32)
    assert _call_forward(L, d) in (lily.LILY_ERR_CUDA, lily.LILY_ERR_ARCH)


def test_host_graph_switch_and_host_entry_arguments(L):
    """The end-to-end call's graph-cache switch returns the previous setting
    (with the cache empty it makes no CUDA call), and the host-buffer entry
    rejects missing host buffers before any copy or launch."""
    first = L.lily_moe_host_graphs(0)
    try:
        assert first in (0, 1)
        assert L.lily_moe_host_graphs(0) == 0
        assert L.lily_moe_host_graphs(1) == 0
        assert L.lily_moe_host_graphs(1) == 1
    finally:
        L.lily_moe_host_graphs(1)
    d = lily.make_dims(64, 512, 32, 4, 128, 32)
    wt = _lib.Weights(*([256] * 11))
    rt = _lib.Routing(*([256] * 9))
    args = dict(x_host=16, x_dev=16, y_dev=16, y_host=16)
    for missing in ("x_host", "y_host"):
        a = dict(args, **{missing: None})
        rc = L.lily_moe_forward_host(ctypes.byref(d), a["x_host"], a["x_dev"], ctypes.byref(wt),
                                     ctypes.byref(rt), a["y_dev"], a["y_host"], 16, 1 << 40, None)
        assert rc == lily.LILY_ERR_INVALID_ARG, missing


def test_route_wait_limit_setter_returns_previous(L):
    """The routing wait limit defaults to 2 s and the setter returns the
    previous value (host state only: no CUDA call)."""
    prev = lily.lily_moe_set_route_wait_ns(12345)
    try:
        assert prev == 2_000_000_000
        assert lily.lily_moe_set_route_wait_ns(0) == 12345
    finally:
        assert lily.lily_moe_set_route_wait_ns(prev) == 0


def test_static_decode_refuses_rows_before_size(L):
    """The static-scratch decode refuses T > 8 as a shape error even when the
    dims would also exceed its fixed scratch, and oversized dims as a
    workspace error, before any CUDA call."""
    w = _lib.Weights(*([256] * 11))
    r = _lib.Routing(*([256] * 9))
    many = lily.make_dims(9, 4096, 256, 8, 4096, 128)
    assert L.lily_moe_decode_static(ctypes.byref(many), 256, ctypes.byref(w), ctypes.byref(r),
                                    256, None) == lily.LILY_ERR_UNSUPPORTED_SHAPE
    big = lily.make_dims(8, 4096, 256, 8, 4096, 128)
    assert L.lily_moe_decode_static(ctypes.byref(big), 256, ctypes.byref(w), ctypes.byref(r),
                                    256, None) == lily.LILY_ERR_WORKSPACE_TOO_SMALL


def test_router_split_arguments(L):
    """The one-time router split reports its size and checks its arguments
    before any CUDA call; a misaligned split in the weights is refused."""
    assert L.lily_moe_router_split_bytes(256, 2048) == 3 * 256 * 2048 * 2
    assert L.lily_moe_router_split_bytes(0, 2048) == 0
    assert L.lily_moe_router_split(None, 256, 2048, 256, None) == lily.LILY_ERR_INVALID_ARG
    assert L.lily_moe_router_split(256, 256, 2048, None, None) == lily.LILY_ERR_INVALID_ARG
    assert L.lily_moe_router_split(256, 257, 2048, 256, None) == lily.LILY_ERR_INVALID_ARG
    assert L.lily_moe_router_split(256, 256, 2000, 256, None) == lily.LILY_ERR_UNSUPPORTED_SHAPE
    assert L.lily_moe_router_split(264, 256, 2048, 256, None) == lily.LILY_ERR_MISALIGNED
    assert L.lily_moe_router_split(256, 256, 2048, 264, None) == lily.LILY_ERR_MISALIGNED
    d = lily.make_dims(64, 512, 32, 4, 128, 32)
    wt = _lib.Weights(*([256] * 11))
    wt.router_w_split = 264
    rt = _lib.Routing(*([256] * 9))
    assert L.lily_moe_forward(ctypes.byref(d), 16, ctypes.byref(wt), ctypes.byref(rt), 16, 16,
                              1 << 40, None) == lily.LILY_ERR_MISALIGNED
