"""Stacked decode step (lily_moe_stack_decode) vs the oracle.

One call runs n_layers pre-norm MoE layers on T = 1..8 rows: each layer's
router applies unit RMSNorm and the bf16 rounding itself, routes, and the
expert GEMVs add the layer output into the fp32 residual, all chained on the
device.  Every layer is checked on every row: the oracle takes the GPU's own
input of that layer (traced), applies RMSNorm and the bf16 rounding, scores
the router in fp64 (compared with the GPU's traced logits), routes from the
GPU's fp32 logits, and its layer output is compared with x_{l+1} - x_l.  An
RMSNorm output within the kernel's fp32 error of a bf16 rounding boundary may
round either way; the logit bound allows for exactly those elements.
"""
import numpy as np
import pytest
import torch

import oracle
import w4_grouped_gemm_gb300 as lily
from w4_grouped_gemm_gb300 import synth

from gpu_util import LOGIT_REL, assert_layer_close

pytestmark = pytest.mark.gpu

EPS = 1e-6


def _bf16_round_bits(a64):
    t = torch.from_numpy(np.asarray(a64, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# Relative distance from a bf16 rounding boundary within which either
# neighbour is a correct rounding of an RMSNorm output: the kernel forms the
# row's scale in fp32 (a sum of d squares in a tree of at most ~24 roundings,
# a square root and a reciprocal), about 1e-6 relative at worst.
NEAR_TIE_REL = 2e-6


def _bf16_values(a64):
    t = torch.from_numpy(np.asarray(a64, np.float32)).to(torch.bfloat16)
    return t.float().numpy().astype(np.float64)


def _near_tie_slack(x64, w):
    """The most each logit ([T][E]) can move when the RMSNorm outputs that lie
    within NEAR_TIE_REL of a bf16 rounding boundary round the other way:
    sum over those elements of |w| times the bf16 step between the two
    neighbours (zero everywhere else)."""
    step = np.abs(_bf16_values(x64 * (1 + NEAR_TIE_REL)) -
                  _bf16_values(x64 * (1 - NEAR_TIE_REL)))
    return step @ np.abs(np.asarray(w, np.float64)).T


def _used_experts(experts, ids, E):
    """The experts the rows use plus the shared expert (last), copied to the
    host, and the ids renumbered into that compact set."""
    used = np.unique(ids)
    idx = torch.tensor(list(used) + [E], dtype=torch.long, device=experts["gate_q"].device)
    sub = {n: t.index_select(0, idx) for n, t in experts.items()}
    remap = np.full(E, -1, np.int32)
    remap[used] = np.arange(len(used), dtype=np.int32)
    return synth.experts_to_numpy(sub), remap[ids]


def _run(T, n_layers, d, E, k, F, seed):
    dev = torch.device("cuda")
    layers = []
    for l in range(n_layers):
        wr, br = synth.make_router(E, d, seed + 10 * l + 1, dev)
        ex = synth.make_experts(E, d, F, seed + 10 * l + 2, dev)
        layers.append(lily.LayerWeights(wr, br, ex))
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    x = torch.randn(T, d, generator=g, device=dev, dtype=torch.float32)
    dims = lily.make_dims(T, d, E, k, F, 128)
    ws = lily.alloc_workspace(lily.lily_moe_stack_workspace_bytes(dims), dev)
    trace_x = torch.empty(n_layers, T, d, dtype=torch.float32, device=dev)
    trace_l = torch.empty(n_layers, T, E, dtype=torch.float32, device=dev)
    lily.lily_moe_stack_decode(dims, x, layers, EPS, trace_x, trace_l, ws)
    torch.cuda.synchronize()
    assert lily.lily_moe_status(ws) == 0
    return layers, x, trace_x, trace_l


def _check_stack(T, n_layers, d, E, k, F, seed):
    layers, x, tx, tl = _run(T, n_layers, d, E, k, F, seed)
    assert bool(torch.isfinite(x).all())
    xs = [tx[l].cpu().numpy() for l in range(n_layers)] + [x.cpu().numpy()]
    worst = 0.0
    for l in range(n_layers):
        xin, xout = xs[l], xs[l + 1]
        x64 = oracle.rmsnorm(xin, EPS)
        xn = _bf16_round_bits(x64)
        logits = tl[l].cpu().numpy()
        w = layers[l].router_w.cpu().numpy()
        L64, A = oracle.router_logits(xn, w, None)
        slack = _near_tie_slack(x64, w)
        assert np.all(np.abs(logits - L64) <= LOGIT_REL * A + slack + 1e-30), f"layer {l}: logits"
        ro = oracle.route(logits, k, 128)
        w, ids = _used_experts(layers[l].experts, ro["ids"], E)
        ref = oracle.moe_rows(xn, w, ids, ro["gates"], np.arange(T))
        got = xout.astype(np.float64) - xin.astype(np.float64)
        mx, _ = assert_layer_close(got, ref, f"stack decode layer {l}")
        worst = max(worst, mx)
    return worst


def test_stack_decode_small_40_layers(oracle_lib):
    _check_stack(3, 40, 512, 32, 4, 128, seed=9000)


def test_stack_decode_full_size_t1_40_layers(oracle_lib):
    """Batch-1 decode through 40 full-size layers (d 2048, 256 experts top-8
    + shared, F 512): every layer on its row."""
    _check_stack(1, 40, 2048, 256, 8, 512, seed=9100)


@pytest.mark.parametrize("T", [5, 8])
def test_stack_decode_full_size_verify_rows(oracle_lib, T):
    """Speculative-verify batches through 6 full-size layers."""
    _check_stack(T, 6, 2048, 256, 8, 512, seed=9200 + T)
