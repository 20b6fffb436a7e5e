"""Stacked prefill (pre-norm MoE layers, fp32 residual, bounded chunks) vs
the oracle.

Rows of a MoE-only stack are independent, so each layer is checked on
sampled rows: the oracle takes the GPU's own input of that layer (traced),
applies unit RMSNorm and the bf16 rounding, routes from the GPU's traced fp32
logits, and its layer output is compared with x_{l+1} - x_l.
"""
import numpy as np
import pytest
import torch

import oracle
import w4_grouped_gemm_gb300 as lily
from w4_grouped_gemm_gb300 import synth

from gpu_util import assert_layer_close

pytestmark = pytest.mark.gpu

EPS = 1e-6


def _bf16_round_bits(a64):
    t = torch.from_numpy(np.asarray(a64, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _run_stack(T_total, chunk, n_layers, d, E, k, F, tile_rows, seed):
    dev = torch.device("cuda")
    shape = synth.LayerShape(chunk, d, E, k, F)
    layers = []
    for l in range(n_layers):
        wr, br = synth.make_router(E, d, seed + 10 * l + 1, dev)
        ex = synth.make_experts(E, d, F, seed + 10 * l + 2, dev)
        layers.append(lily.LayerWeights(wr, br, ex))
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    x0 = torch.randn(T_total, d, generator=g, device=dev, dtype=torch.float32)
    x = x0.clone()
    dims = lily.make_dims(chunk, d, E, k, F, tile_rows)
    ws = lily.alloc_workspace(lily.lily_moe_stack_workspace_bytes(dims), dev)
    trace_x = torch.empty(n_layers, T_total, d, dtype=torch.float32, device=dev)
    trace_l = torch.empty(n_layers, T_total, E, dtype=torch.float32, device=dev)
    lily.lily_moe_stack_prefill(dims, x, layers, EPS, trace_x, trace_l, ws)
    torch.cuda.synchronize()
    assert lily.lily_moe_status(ws) == 0
    return shape, layers, x, trace_x, trace_l


def _check_layer(layer, xin, xout, logits, k, rows):
    """Oracle layer on rows of the GPU's layer input; returns the errors."""
    xn = _bf16_round_bits(oracle.rmsnorm(xin[rows], EPS))
    ro = oracle.route(logits[rows], k, 128)
    w = synth.experts_to_numpy(layer.experts)
    ref = oracle.moe_rows(xn, w, ro["ids"], ro["gates"], np.arange(len(rows)))
    got = xout[rows].astype(np.float64) - xin[rows].astype(np.float64)
    return assert_layer_close(got, ref, "stack layer")


def test_stack_small_full_rows(oracle_lib):
    T_total, chunk, L = 96, 32, 3
    shape, layers, x, tx, tl = _run_stack(T_total, chunk, L, 512, 32, 4, 128, 32, seed=5000)
    xs = [tx[l].cpu().numpy() for l in range(L)] + [x.cpu().numpy()]
    for l in range(L):
        _check_layer(layers[l], xs[l], xs[l + 1], tl[l].cpu().numpy(), 4, np.arange(T_total))


def test_stack_40_layers_8192_tokens(oracle_lib):
    """The full stacked workload: 40 layers, 8192 tokens in chunks of 2048,
    every layer checked on 4 sampled rows (one per chunk)."""
    T_total, chunk, L = 8192, 2048, 40
    shape, layers, x, tx, tl = _run_stack(T_total, chunk, L, 2048, 256, 8, 512, 128, seed=6000)
    assert bool(torch.isfinite(x).all())
    rng = np.random.default_rng(0)
    worst = 0.0
    for l in range(L):
        rows = np.array([c * chunk + rng.integers(chunk) for c in range(T_total // chunk)])
        xin = tx[l][rows].cpu().numpy()
        xout = (tx[l + 1][rows] if l + 1 < L else x[rows]).cpu().numpy()
        mx, _ = _check_layer(layers[l], xin, xout, tl[l][rows].cpu().numpy(), 8,
                             np.arange(len(rows)))
        worst = max(worst, mx)
    rms = float(x.pow(2).mean().sqrt())
    assert 1.0 < rms < 1e4, rms   # the pre-norm stack stays bounded
