"""lily_moe_decode_static: the decode layer for callers that cannot allocate.

Its scratch lives in a fixed array inside the library instead of a caller
workspace.  Called through the C ABI twice in a row (different inputs, so the
second call starts from the first call's leftovers), each output must match
lily_moe_decode -- the entry point with a caller workspace -- within the layer
tolerance the other parity tests use.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import w4_grouped_gemm_gb300 as lily
from w4_grouped_gemm_gb300 import _lib, synth

from gpu_util import Layer, assert_layer_close

pytestmark = pytest.mark.gpu


def _decode_static(L: Layer, y: torch.Tensor) -> int:
    lib = lily.lib()
    return lib.lily_moe_decode_static(ctypes.byref(L.dims), L.x.data_ptr(), ctypes.byref(L.w.c),
                                      ctypes.byref(L.r.c), y.data_ptr(),
                                      torch.cuda.current_stream().cuda_stream)


def test_decode_static_matches_decode_two_calls(oracle_lib):
    cases = [Layer(synth.LayerShape(5, 2048, 256, 8, 512), seed=7100, tile_rows=128),
             Layer(synth.LayerShape(2, 2048, 256, 8, 512), seed=7200, tile_rows=128)]
    for L in cases:
        y_static = torch.full_like(L.y, float("nan"))
        rc = _decode_static(L, y_static)
        assert rc == lily.LILY_OK, lily.strerror(rc)
        torch.cuda.synchronize()
        ids_static = L.r.topk_ids.clone()
        ref = L.decode().double().cpu().numpy()          # caller-workspace entry point
        assert torch.equal(ids_static, L.r.topk_ids)
        assert L.status() == 0
        assert_layer_close(y_static.double().cpu().numpy(), ref, f"static T={L.shape.T}")


def test_decode_static_refuses_oversized_dims(oracle_lib):
    dims = lily.make_dims(8, 4096, 256, 8, 4096, 128)
    assert lily.lily_moe_workspace_bytes(dims) > (1 << 20)
    lib = lily.lib()
    w = _lib.Weights(*([256] * 11))
    r = _lib.Routing(*([256] * 9))
    rc = lib.lily_moe_decode_static(ctypes.byref(dims), 256, ctypes.byref(w), ctypes.byref(r), 256,
                                    None)
    assert rc == lily.LILY_ERR_WORKSPACE_TOO_SMALL
