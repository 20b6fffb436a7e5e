"""Whole-layer parity, CUDA path vs the FP64 oracle.

The oracle routes from the GPU's own fp32 logits (routing parity is tested
bit-exact separately), so a near-tie can never make the two sides pick
different experts.  The fp32 layer output must meet max|err|/rms <= 2e-2 and
mean|err|/mean|ref| <= 5e-3; the bf16 output is that fp32 output rounded once.
"""
import numpy as np
import pytest
import torch

import oracle
import w4_grouped_gemm_gb300 as lily
from w4_grouped_gemm_gb300 import synth

from gpu_util import Layer, assert_layer_close, assert_routing_equal

pytestmark = pytest.mark.gpu


def _check_forward(L, rows=None, decode=False):
    (L.decode if decode else L.forward)()
    assert L.status() == 0
    gpu = L.r.host()
    ro = oracle.route(gpu["logits"], L.shape.k, L.dims.tile_rows)
    assert_routing_equal(gpu, ro, L.shape.T, L.shape.k)
    rows = np.arange(L.shape.T) if rows is None else np.asarray(rows)
    ref = L.oracle_rows(rows, ro)
    got = L.y.float().cpu().numpy()[rows]
    return assert_layer_close(got, ref, f"T={L.shape.T} BM={L.dims.tile_rows}")


# ------------------------------------------------------------ full-layer, small

@pytest.mark.parametrize("bm", [16, 32, 64, 128])
def test_small_layer_all_tile_rows(oracle_lib, bm):
    _check_forward(Layer(synth.SHAPES["small"], seed=1000, tile_rows=bm))


@pytest.mark.parametrize("shape,bm", [
    (synth.LayerShape(37, 256, 16, 3, 128), 32),      # ragged tiles everywhere
    (synth.LayerShape(130, 384, 24, 5, 256), 64),     # 2 F slices, 3 d slices
    (synth.LayerShape(9, 512, 32, 4, 128), 32),       # smallest prefill T
    (synth.LayerShape(257, 128, 8, 8, 128), 128),     # E == k: every expert chosen
    (synth.LayerShape(150, 256, 8, 2, 4096), 128),    # largest F: a 3-stage down ring
    (synth.LayerShape(70, 4096, 4, 2, 128), 64),      # largest d: one gate/up scale table
])
def test_ragged_layers(oracle_lib, shape, bm):
    _check_forward(Layer(shape, seed=shape.T * 7, tile_rows=bm))


def test_all_tokens_one_expert(oracle_lib):
    """A huge router bias sends every token to expert 5 first: one expert with
    T rows spans many tiles; most experts are empty."""
    shape = synth.LayerShape(300, 512, 32, 2, 128)
    b = torch.zeros(32, dtype=torch.float32, device="cuda")
    b[5] = 100.0
    b[9] = 50.0
    L = Layer(shape, seed=55, tile_rows=64, router_b=b)
    _check_forward(L)
    counts = L.r.counts.cpu().numpy()
    assert counts[5] == 300 and counts[9] == 300 and counts.sum() == 600


def test_identical_experts_closed_form(oracle_lib):
    """Every routed expert and the shared expert identical: y = 2 FFN(x) on
    the GPU too (gates sum to 1), checked against the oracle's closed form."""
    shape = synth.LayerShape(64, 512, 16, 4, 128)
    one = synth.make_experts(0, shape.d, shape.F, seed=77, device="cuda")
    experts = {n: t.expand(shape.E + 1, *t.shape[1:]).contiguous() for n, t in one.items()}
    L = Layer(shape, seed=78, tile_rows=32, experts=experts)
    L.forward()
    npone = synth.experts_to_numpy(one)
    ref = 2.0 * _dense_ffn(npone, synth.bf16_bits(L.x))
    assert_layer_close(L.y.float().cpu().numpy(), ref, "identical experts")


def _dense_ffn(npw, xbits):
    x = (xbits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    Wg = oracle.dequant(npw["gate_q"][0], npw["gate_s"][0], npw["gate_b"][0])
    Wu = oracle.dequant(npw["up_q"][0], npw["up_s"][0], npw["up_b"][0])
    Wd = oracle.dequant(npw["down_q"][0], npw["down_s"][0], npw["down_b"][0])
    g = x @ Wg.T
    h = g / (1.0 + np.exp(-g)) * (x @ Wu.T)
    return h @ Wd.T


# ------------------------------------------------------------ full-size configs

def test_prefill512_sampled_rows(oracle_lib):
    L = Layer(synth.SHAPES["prefill512"], seed=2000, tile_rows=128)
    rows = np.random.default_rng(1).choice(512, 40, replace=False)
    _check_forward(L, rows)


def test_prefill2048_zipf_sampled_rows(oracle_lib):
    L = Layer(synth.SHAPES["prefill2048_zipf"], seed=3000, tile_rows=128, zipf_s=1.1)
    rows = np.random.default_rng(2).choice(2048, 32, replace=False)
    _check_forward(L, rows)
    counts = L.r.counts.cpu().numpy()
    assert (counts == 0).any() and counts.max() > 256


def test_prefill2048_uniform_sampled_rows_bm64(oracle_lib):
    L = Layer(synth.SHAPES["prefill2048_zipf"], seed=3100, tile_rows=64)
    rows = np.random.default_rng(3).choice(2048, 24, replace=False)
    _check_forward(L, rows)


def test_prefill2048_uniform_sampled_rows_bm128(oracle_lib):
    L = Layer(synth.SHAPES["prefill2048_zipf"], seed=3200, tile_rows=128)
    rows = np.random.default_rng(4).choice(2048, 24, replace=False)
    _check_forward(L, rows)


def test_prefill512_bm16_sampled_rows(oracle_lib):
    L = Layer(synth.SHAPES["prefill512"], seed=2100, tile_rows=16)
    rows = np.random.default_rng(5).choice(512, 24, replace=False)
    _check_forward(L, rows)


def test_prefill8192_one_call_sampled_rows(oracle_lib):
    """The unchunked long-prompt layer: one call of T = 8192 tokens (weights
    read once), bit-exact routing and 64 sampled rows spread over the whole
    range (one from each block of 128 tokens) against the oracle."""
    L = Layer(synth.LayerShape(8192, 2048, 256, 8, 512), seed=3300, tile_rows=128)
    rng = np.random.default_rng(6)
    rows = np.arange(0, 8192, 128) + rng.integers(0, 128, 64)
    _check_forward(L, rows)


@pytest.mark.parametrize("T,bm", [(256, 64), (2048, 128)])
def test_forward_repeat_is_bit_identical(oracle_lib, T, bm):
    """Two calls on the same workspace give the same routing and the same
    output bits: every sum of the layer has a fixed order (the combine adds
    each token's rows in slot order)."""
    L = Layer(synth.LayerShape(T, 1024, 64, 8, 256), seed=91, tile_rows=bm)
    y1 = L.forward().clone()
    ids1 = L.r.topk_ids.clone()
    y2 = L.forward()
    assert torch.equal(ids1, L.r.topk_ids)
    assert torch.equal(y1, y2)


# ------------------------------------------------------------ decode path

@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 8])
def test_decode_full_size(oracle_lib, T):
    _check_forward(Layer(synth.LayerShape(T, 2048, 256, 8, 512), seed=4000 + T, tile_rows=128),
                   decode=True)


def test_decode_small_shape(oracle_lib):
    _check_forward(Layer(synth.LayerShape(3, 512, 32, 4, 128), seed=4100, tile_rows=32),
                   decode=True)


def test_decode_matches_forward(oracle_lib):
    """Decode (GEMV) and prefill (grouped GEMM) paths agree on T = 8."""
    L = Layer(synth.LayerShape(8, 1024, 64, 8, 256), seed=4200, tile_rows=32)
    yd = L.decode().float().clone()
    yf = L.forward().float()
    rel = (yd - yf).abs().max().item() / yf.pow(2).mean().sqrt().item()
    assert rel < 5e-3


def test_forward_host_entry(oracle_lib):
    """The host-buffer entry point gives the same result as the device one."""
    L = Layer(synth.LayerShape(64, 512, 32, 4, 128), seed=4300, tile_rows=32)
    ydev = L.forward().clone()
    xh = L.x.cpu().pin_memory()
    yh = torch.empty(64, 512, dtype=L.y.dtype).pin_memory()
    xd = torch.empty_like(L.x)
    yd = torch.empty_like(L.y)
    lily.lily_moe_forward_host(L.dims, xh, xd, L.w, L.r, yd, yh, L.ws)
    assert torch.equal(yh, ydev.cpu())


def test_forward_host_async_two_streams(oracle_lib):
    """Two host-buffer calls in flight on two streams, each with its own
    staging, routing buffers, workspace and host buffers: once a stream is
    synchronised its host output equals the device entry point's result for
    that call's input (each set's first call runs eagerly, later ones replay
    its graph), and a set is refilled only after its stream has finished."""
    T, d = 64, 512
    L = Layer(synth.LayerShape(T, d, 32, 4, 128), seed=4400, tile_rows=32)
    g = torch.Generator().manual_seed(4401)
    xs = [(torch.randn(T, d, generator=g) * (1.0 + c)).to(torch.bfloat16) for c in range(6)]
    refs = []
    for x in xs:  # device entry point, before the sets share L's buffers
        L.x.copy_(x)
        refs.append(L.forward().cpu().clone())
    lily.lily_moe_host_graphs(True)
    dev = L.x.device
    sets = []
    for j in range(2):
        sets.append({
            "r": L.r if j == 0 else lily.RoutingBuffers(L.dims, dev),
            "ws": L.ws if j == 0 else lily.alloc_workspace(lily.lily_moe_workspace_bytes(L.dims),
                                                           dev),
            "xh": torch.empty(T, d, dtype=torch.bfloat16).pin_memory(),
            "yh": torch.empty(T, d, dtype=L.y.dtype).pin_memory(),
            "xd": torch.empty_like(L.x), "yd": torch.empty_like(L.y),
            "s": torch.cuda.Stream(device=dev), "call": None})
    for c, x in enumerate(xs):
        b = sets[c % 2]
        b["s"].synchronize()
        if b["call"] is not None:
            assert torch.equal(b["yh"], refs[b["call"]]), f"call {b['call']}"
        b["xh"].copy_(x)
        b["yh"].fill_(float("nan"))
        lily.lily_moe_forward_host_async(L.dims, b["xh"], b["xd"], L.w, b["r"], b["yd"], b["yh"],
                                         b["ws"], b["s"])
        b["call"] = c
    for b in sets:
        b["s"].synchronize()
        assert torch.equal(b["yh"], refs[b["call"]]), f"call {b['call']}"
        assert lily.lily_moe_status(b["ws"]) == 0


@pytest.mark.parametrize("T", [64, 5])
@pytest.mark.parametrize("pinned", [True, False])
def test_forward_host_graph_cache(oracle_lib, T, pinned):
    """Repeated host-buffer calls with one argument set: the first runs
    eagerly and captures a graph, the next ones replay it.  The host input
    changes between calls, so a replay that read stale data fails; every call
    must match the device entry point on the same x."""
    shape = synth.LayerShape(T, 512, 32, 4, 128)
    L = Layer(shape, seed=4310 + T, tile_rows=32)
    run = L.decode if T <= 8 else L.forward
    lily.lily_moe_host_graphs(True)
    xh = torch.empty(T, 512, dtype=torch.bfloat16)
    yh = torch.empty(T, 512, dtype=L.y.dtype)
    if pinned:
        xh, yh = xh.pin_memory(), yh.pin_memory()
    xd = torch.empty_like(L.x)
    yd = torch.empty_like(L.y)
    g = torch.Generator().manual_seed(77 + T)
    try:
        for call in range(4):
            x = (torch.randn(T, 512, generator=g) * (1.0 + call)).to(torch.bfloat16)
            L.x.copy_(x)
            yref = run().float().cpu().clone()
            xh.copy_(x)
            yh.fill_(float("nan"))
            lily.lily_moe_forward_host(L.dims, xh, xd, L.w, L.r, yd, yh, L.ws)
            assert L.status() == 0
            rel = (yh.float() - yref).abs().max().item() / yref.pow(2).mean().sqrt().item()
            assert rel < 1e-4, f"call {call}: rel {rel}"
        # profiling forces the eager path: same result
        lily.lily_moe_profile_enable(True)
        yh.fill_(float("nan"))
        lily.lily_moe_forward_host(L.dims, xh, xd, L.w, L.r, yd, yh, L.ws)
        lily.lily_moe_profile_read()
        lily.lily_moe_profile_enable(False)
        rel = (yh.float() - yref).abs().max().item() / yref.pow(2).mean().sqrt().item()
        assert rel < 1e-4, f"eager call: rel {rel}"
    finally:
        lily.lily_moe_profile_enable(False)
        lily.lily_moe_host_graphs(True)


@pytest.mark.parametrize("decode", [False, True])
def test_bf16_output_is_rounded_fp32_output(oracle_lib, decode):
    """out_dtype = bf16 gives exactly the fp32 output rounded once to bf16, for
    both paths (the fp32 sums are the same bits on every run)."""
    shape = synth.LayerShape(8 if decode else 96, 512, 32, 4, 128)
    Lf = Layer(shape, seed=4400, tile_rows=32)
    Lb = Layer(shape, seed=4400, tile_rows=32, out_dtype=lily.LILY_DTYPE_BF16)
    yf = Lf.decode() if decode else Lf.forward()
    yb = Lb.decode() if decode else Lb.forward()
    assert Lb.y.dtype == torch.bfloat16
    assert torch.equal(yb, yf.to(torch.bfloat16))


def test_experts_entry_with_host_routing(oracle_lib):
    """lily_moe_experts on routing built on the host (the oracle's routing of
    the GPU's fp32 logits, uploaded) reproduces lily_moe_forward bit for bit:
    the same routing and the same kernels, whose sums have a fixed order."""
    L = Layer(synth.SHAPES["small"], seed=4242, tile_rows=32)
    y_fwd = L.forward().clone()
    ro = L.oracle_route()
    r2 = lily.RoutingBuffers(L.dims)
    dev = r2.perm.device

    def up(a, like):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev, like.dtype).reshape(like.shape)

    r2.logits.copy_(L.r.logits)
    r2.topk_gates.copy_(L.r.topk_gates)  # fp32 gates as the GPU computed them
    r2.topk_ids.copy_(up(ro["ids"], r2.topk_ids))
    r2.counts.copy_(up(ro["counts"], r2.counts))
    r2.offsets.copy_(up(ro["offsets"], r2.offsets))
    r2.perm.copy_(up(ro["perm"], r2.perm))
    r2.inv_perm.copy_(up(ro["inv"], r2.inv_perm))
    r2.block_map.copy_(up(ro["block_map"], r2.block_map))
    r2.n_tiles.fill_(ro["n_tiles"])
    y2 = torch.empty_like(y_fwd)
    lily.lily_moe_experts(L.dims, L.x, L.w, r2, y2, L.ws)
    torch.cuda.synchronize()
    assert L.status() == 0
    assert torch.equal(y2, y_fwd)


def test_experts_entry_flags_bad_perm(oracle_lib):
    """Out-of-range perm entries are clamped and flagged, never read out of
    bounds."""
    L = Layer(synth.SHAPES["small"], seed=4343, tile_rows=32)
    L.forward()
    assert L.status() == 0
    L.r.perm[3] = 1 << 20
    y2 = torch.empty_like(L.y)
    lily.lily_moe_experts(L.dims, L.x, L.w, L.r, y2, L.ws)
    torch.cuda.synchronize()
    assert L.status() & lily.LILY_STATUS_BAD_TILE
