"""Device error paths: a bounded wait that gives up, and values beyond the fp16
range of the tensor-core operands.  Neither traps: each sets a status bit that
lily_moe_status() returns, and the workspace stays usable afterwards."""
import numpy as np
import pytest
import torch

import oracle
import w4_grouped_gemm_gb300 as lily
from w4_grouped_gemm_gb300 import synth

from gpu_util import Layer, assert_routing_equal

pytestmark = pytest.mark.gpu


def _route_and_check(L):
    lily.lily_moe_route(L.dims, L.x, None, L.w, L.r, L.ws)
    torch.cuda.synchronize()
    assert L.status() == 0
    gpu = L.r.host()
    ro = oracle.route(gpu["logits"], L.shape.k, L.dims.tile_rows)
    assert_routing_equal(gpu, ro, L.shape.T, L.shape.k)


def test_route_barrier_timeout_then_recovers(oracle_lib):
    """A zero wait limit makes the blocks that wait at the routing kernel's
    grid barrier give up at once: the call sets LILY_STATUS_TIMEOUT and
    returns.  With the limit restored, the same workspace (its status read,
    which also clears the barrier counters) and a fresh one route bit-exactly."""
    shape = synth.LayerShape(8192, 256, 64, 8, 128)   # 256 routing blocks
    L = Layer(shape, seed=8100, tile_rows=128)
    prev = lily.lily_moe_set_route_wait_ns(0)
    try:
        lily.lily_moe_route(L.dims, L.x, None, L.w, L.r, L.ws)
        torch.cuda.synchronize()
    finally:
        assert lily.lily_moe_set_route_wait_ns(prev) == 0
    assert prev == 2_000_000_000
    assert L.status() & lily.LILY_STATUS_TIMEOUT
    _route_and_check(L)                                        # same workspace
    L2 = Layer(shape, seed=8100, tile_rows=128)
    _route_and_check(L2)                                       # fresh workspace
    assert torch.equal(L.r.perm, L2.r.perm)


@pytest.mark.parametrize("T", [64, 1])
def test_f16_range_flagged(oracle_lib, T):
    """A bf16 input of 1e5 is outside the fp16 operand range: prefill flags it
    when the token rows are converted, decode when silu(g)*u overflows fp16 in
    H.  A normal input on the same workspace afterwards raises nothing."""
    shape = synth.LayerShape(T, 512, 32, 4, 128)
    L = Layer(shape, seed=8200 + T, tile_rows=32)
    run = L.decode if T <= 8 else L.forward
    x_ok = L.x.clone()
    L.x[T - 1, 7] = 1e5
    run()
    assert L.status() & lily.LILY_STATUS_F16_RANGE
    L.x.copy_(x_ok)
    run()
    assert L.status() == 0
    assert bool(torch.isfinite(L.y).all())
