"""GPU routing vs the oracle: bit-exact ids / histogram / scan / scatter /
block map given the GPU's fp32 logits, gates within 1e-6, logits within the
fp32 accumulation bound."""
import numpy as np
import pytest
import torch

import oracle
import w4_grouped_gemm_gb300 as lily
from w4_grouped_gemm_gb300 import synth

from gpu_util import LOGIT_REL, Layer, assert_routing_equal

pytestmark = pytest.mark.gpu

CASES = [
    # name, shape, tile_rows, zipf
    ("small", synth.LayerShape(32, 512, 32, 4, 128), 32, None),
    ("ragged", synth.LayerShape(37, 256, 16, 3, 128), 32, None),
    ("prefill512", synth.LayerShape(512, 2048, 256, 8, 512), 128, None),
    ("prefill2048_zipf", synth.LayerShape(2048, 2048, 256, 8, 512), 128, 1.1),
    ("decode1", synth.LayerShape(1, 2048, 256, 8, 512), 128, None),
    ("decode5", synth.LayerShape(5, 2048, 256, 8, 512), 128, None),
    ("bm32_2048", synth.LayerShape(2048, 2048, 256, 8, 512), 32, None),
    ("bm64_600", synth.LayerShape(600, 1024, 64, 6, 256), 64, None),
    ("max_tokens", synth.LayerShape(16384, 128, 256, 8, 128), 64, None),
]


@pytest.mark.parametrize("name,shape,bm,zipf", CASES, ids=[c[0] for c in CASES])
def test_route_bitexact(oracle_lib, name, shape, bm, zipf):
    L = Layer(shape, seed=100 + shape.T, tile_rows=bm, zipf_s=zipf)
    lily.lily_moe_route(L.dims, L.x, None, L.w, L.r, L.ws)
    torch.cuda.synchronize()
    assert L.status() == 0
    gpu = L.r.host()
    ro = oracle.route(gpu["logits"], shape.k, bm)
    assert ro["n_nan"] == 0
    assert_routing_equal(gpu, ro, shape.T, shape.k)
    # logits against double, on a sample of rows for the big cases
    rows = np.arange(shape.T) if shape.T <= 64 else np.random.default_rng(0).choice(
        shape.T, 48, replace=False)
    xb = synth.bf16_bits(L.x)[rows]
    wr = L.inp["router_w"].cpu().numpy()
    br = None if L.inp["router_b"] is None else L.inp["router_b"].cpu().numpy()
    Ld, A = oracle.router_logits(xb, wr, br)
    err = np.abs(gpu["logits"][rows].astype(np.float64) - Ld)
    assert np.all(err <= LOGIT_REL * A + 1e-7), float((err / (A + 1e-30)).max())


def test_route_zipf_has_empty_and_big_groups(oracle_lib):
    L = Layer(synth.SHAPES["prefill2048_zipf"], seed=3000, tile_rows=128, zipf_s=1.1)
    lily.lily_moe_route(L.dims, L.x, None, L.w, L.r, L.ws)
    counts = L.r.counts.cpu().numpy()
    assert (counts == 0).sum() > 0 and counts.max() > 512


@pytest.mark.parametrize("T,E,k,bm", [(64, 8, 3, 32), (200, 256, 8, 32), (3, 4, 4, 32)])
def test_route_from_given_logits_with_ties(oracle_lib, T, E, k, bm):
    """Integer-valued logits force many ties; -0/+0 and a NaN are included."""
    rng = np.random.default_rng(T)
    Lg = rng.integers(-3, 4, size=(T, E)).astype(np.float32)
    Lg[0, 0] = -0.0
    Lg[0, 1] = 0.0
    dims = lily.make_dims(T, 512, E, k, 128, bm)
    r = lily.RoutingBuffers(dims)
    ws = lily.alloc_workspace(lily.lily_moe_workspace_bytes(dims))
    lt = torch.from_numpy(Lg).cuda()
    lily.lily_moe_route(dims, None, lt, None, r, ws)
    torch.cuda.synchronize()
    assert lily.lily_moe_status(ws) == 0
    gpu = r.host()
    assert np.array_equal(gpu["logits"], Lg)
    assert_routing_equal(gpu, oracle.route(Lg, k, bm), T, k)
    # NaN logit: flagged on the device, other tokens unaffected
    Lg2 = Lg.copy()
    Lg2[T - 1, E - 1] = np.nan
    lily.lily_moe_route(dims, None, torch.from_numpy(Lg2).cuda(), None, r, ws)
    assert lily.lily_moe_status(ws) & lily.LILY_STATUS_NAN_LOGIT
    assert lily.lily_moe_status(ws) == 0  # cleared by the read
    gpu2 = r.host()
    ro2 = oracle.route(Lg2, k, bm)
    assert np.array_equal(gpu2["topk_ids"], ro2["ids"])


def test_route_repeated_calls_reuse_workspace(oracle_lib):
    """The grid barrier and counters return to a consistent state."""
    L = Layer(synth.LayerShape(300, 512, 64, 4, 128), seed=7, tile_rows=64)
    first = None
    for _ in range(5):
        lily.lily_moe_route(L.dims, L.x, None, L.w, L.r, L.ws)
        torch.cuda.synchronize()
        h = L.r.host()
        if first is None:
            first = h
        for n in ("topk_ids", "perm", "block_map", "counts"):
            assert np.array_equal(h[n], first[n])
    assert L.status() == 0
