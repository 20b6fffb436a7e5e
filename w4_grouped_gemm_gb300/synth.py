"""Seeded synthetic inputs for the W4 MoE expert layer.

This module only draws random numbers: it holds none of the layer's arithmetic.
Both the CUDA path (through the benchmark and tests) and the CPU oracle consume
the tensors it makes, so it is the one module the two sides share.

Distributions (the workload of the Lily pages, shapes chosen by this project):
  x        bf16 ~ N(0, 1)                       [T][d]
  router W fp32 ~ N(0, 0.02^2)                  [E][d]
  router b fp32, optional: skew_s * -ln(e + 1)  [E]   (log of a Zipf(s) pmf
           over rank e+1; only used for the skewed-routing workload)
  q        uniform over 0..15, two codes per byte (every byte uniform 0..255)
  scale    bf16 ~ U(0.001, 0.01)   one per 64 input-dim weights
  bias     bf16 ~ U(-0.08, 0)      one per 64 input-dim weights
Experts are stored E+1 deep: index E is the always-on shared expert.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

GROUP = 64


@dataclass(frozen=True)
class LayerShape:
    T: int
    d: int
    E: int
    k: int
    F: int


# Named workloads (sizes of the Lily Qwen3.6-35B-A3B-style MoE layer).
SHAPES = {
    "small": LayerShape(T=32, d=512, E=32, k=4, F=128),
    "prefill512": LayerShape(T=512, d=2048, E=256, k=8, F=512),
    "prefill2048_zipf": LayerShape(T=2048, d=2048, E=256, k=8, F=512),
    "decode": LayerShape(T=1, d=2048, E=256, k=8, F=512),
    "stack8192": LayerShape(T=2048, d=2048, E=256, k=8, F=512),
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_x(T: int, d: int, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    return torch.randn(T, d, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def make_router(E: int, d: int, seed: int, device="cpu", zipf_s: float | None = None):
    """(W fp32 [E][d], b fp32 [E] or None)."""
    g = _gen(seed, device)
    w = torch.randn(E, d, generator=g, device=device, dtype=torch.float32) * 0.02
    b = None
    if zipf_s is not None:
        b = torch.tensor([-zipf_s * math.log(e + 1) for e in range(E)], dtype=torch.float32,
                         device=device)
    return w, b


def _uniform_bf16(shape, lo, hi, g, device):
    u = torch.rand(*shape, generator=g, device=device, dtype=torch.float32)
    return (lo + (hi - lo) * u).to(torch.bfloat16)


def make_w4_matrix(n_mat: int, rows: int, cols: int, g: torch.Generator, device):
    """(q uint8 [n_mat][rows][cols/2], scale bf16, bias bf16 [n_mat][rows][cols/64])."""
    q = torch.randint(0, 256, (n_mat, rows, cols // 2), generator=g, device=device,
                      dtype=torch.int32).to(torch.uint8)
    s = _uniform_bf16((n_mat, rows, cols // GROUP), 0.001, 0.01, g, device)
    b = _uniform_bf16((n_mat, rows, cols // GROUP), -0.08, 0.0, g, device)
    return q, s, b


def make_experts(E: int, d: int, F: int, seed: int, device="cpu") -> dict:
    """W4 weights of E routed experts + 1 shared expert (index E)."""
    g = _gen(seed, device)
    gq, gs, gb = make_w4_matrix(E + 1, F, d, g, device)
    uq, us, ub = make_w4_matrix(E + 1, F, d, g, device)
    dq, ds, db = make_w4_matrix(E + 1, d, F, g, device)
    return dict(gate_q=gq, gate_s=gs, gate_b=gb, up_q=uq, up_s=us, up_b=ub,
                down_q=dq, down_s=ds, down_b=db)


def make_layer(shape: LayerShape, seed: int, device="cpu", zipf_s: float | None = None) -> dict:
    """Every input of one layer, drawn from seed, seed+1, seed+2."""
    x = make_x(shape.T, shape.d, seed, device)
    wr, br = make_router(shape.E, shape.d, seed + 1, device, zipf_s)
    w = make_experts(shape.E, shape.d, shape.F, seed + 2, device)
    return dict(x=x, router_w=wr, router_b=br, experts=w)


def bf16_bits(t: torch.Tensor):
    """Raw uint16 bit patterns of a bf16 tensor, as a numpy array (host copy)."""
    import numpy as np
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def experts_to_numpy(w: dict) -> dict:
    out = {}
    for n, t in w.items():
        out[n] = t.detach().cpu().contiguous().numpy() if n.endswith("_q") else bf16_bits(t)
    return out
