"""lily_moe_decode_static: the decode layer for callers that cannot allocate.

Its scratch lives in a fixed array inside the library instead of a caller
workspace.  Called through the C ABI twice in a row (different inputs, so the
second call starts from the first call's leftovers), each output must equal
lily_moe_decode's -- the entry point with a caller workspace -- bit for bit
(both run the same kernels, whose sums have a fixed order), and must meet the
layer tolerance against the FP64 oracle.  No call may allocate device memory:
the torch allocator's counters and the device's free memory stay unchanged
across the calls.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import w4_grouped_gemm_gb300 as lily
from w4_grouped_gemm_gb300 import _lib, synth

from gpu_util import Layer, assert_layer_close, assert_routing_equal

pytestmark = pytest.mark.gpu


def _decode_static(L: Layer, y: torch.Tensor) -> int:
    lib = lily.lib()
    return lib.lily_moe_decode_static(ctypes.byref(L.dims), L.x.data_ptr(), ctypes.byref(L.w.c),
                                      ctypes.byref(L.r.c), y.data_ptr(),
                                      torch.cuda.current_stream().cuda_stream)


def _memory():
    torch.cuda.synchronize()
    return (torch.cuda.memory_allocated(), torch.cuda.memory_reserved(),
            torch.cuda.mem_get_info()[0])


def test_decode_static_matches_decode_two_calls(oracle_lib):
    cases = [Layer(synth.LayerShape(5, 2048, 256, 8, 512), seed=7100, tile_rows=128),
             Layer(synth.LayerShape(2, 2048, 256, 8, 512), seed=7200, tile_rows=128)]
    outs = [torch.full_like(L.y, float("nan")) for L in cases]
    for i, (L, y_static) in enumerate(zip(cases, outs)):
        before = _memory()
        rc = _decode_static(L, y_static)
        assert rc == lily.LILY_OK, lily.strerror(rc)
        after = _memory()
        # nothing allocated by the call: torch's counters exactly; the free
        # device memory also exactly once the array's module is resident
        assert after[:2] == before[:2]
        if i > 0:
            assert after[2] == before[2]
        gpu = L.r.host()
        y_np = y_static.double().cpu().numpy()
        ref = L.decode().double().cpu().numpy()          # caller-workspace entry point
        assert L.status() == 0
        assert np.array_equal(gpu["topk_ids"], L.r.topk_ids.cpu().numpy())
        assert np.array_equal(y_np, ref), f"T={L.shape.T}: static and workspace outputs differ"
        ro = oracle.route(gpu["logits"], L.shape.k, L.dims.tile_rows)
        assert_routing_equal(gpu, ro, L.shape.T, L.shape.k)
        assert_layer_close(y_np, L.oracle_rows(np.arange(L.shape.T), ro), f"static T={L.shape.T}")


def test_decode_static_refuses_bad_dims(oracle_lib):
    lib = lily.lib()
    w = _lib.Weights(*([256] * 11))
    r = _lib.Routing(*([256] * 9))
    big = lily.make_dims(8, 4096, 256, 8, 4096, 128)
    assert lily.lily_moe_workspace_bytes(big) > (1 << 20)
    rc = lib.lily_moe_decode_static(ctypes.byref(big), 256, ctypes.byref(w), ctypes.byref(r), 256,
                                    None)
    assert rc == lily.LILY_ERR_WORKSPACE_TOO_SMALL
    # more rows than decode takes is a shape error, even when it is also too big
    many = lily.make_dims(9, 4096, 256, 8, 4096, 128)
    rc = lib.lily_moe_decode_static(ctypes.byref(many), 256, ctypes.byref(w), ctypes.byref(r), 256,
                                    None)
    assert rc == lily.LILY_ERR_UNSUPPORTED_SHAPE
