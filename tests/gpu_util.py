"""Shared helpers of the GPU parity tests (CUDA path vs the FP64 oracle)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import w4_grouped_gemm_gb300 as lily
from w4_grouped_gemm_gb300 import synth

# Layer-output tolerance (on the fp32 layer output): max|gpu - oracle| /
# rms(oracle) and the mean relative error read as mean|gpu - oracle| /
# mean|oracle|.
MAX_REL_RMS = 2e-2
MEAN_REL = 5e-3
# Gates are fp32 softmax vs the oracle's double: absolute bound.
GATE_TOL = 1e-6
# Router logits: fp32 accumulation of d products; bounded relative to the sum
# of the products' magnitudes.
LOGIT_REL = 1e-5


def layer_errors(got: np.ndarray, ref: np.ndarray):
    got = np.asarray(got, np.float64)
    diff = np.abs(got - ref)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    return float(diff.max() / rms), float(diff.mean() / np.mean(np.abs(ref)))


def assert_layer_close(got, ref, what=""):
    mx, mean = layer_errors(got, ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite GPU output"
    assert mx <= MAX_REL_RMS, f"{what}: max|err|/rms = {mx:.3e}"
    assert mean <= MEAN_REL, f"{what}: mean rel err = {mean:.3e}"
    return mx, mean


class Layer:
    """One seeded layer on the GPU plus the handles the C ABI needs."""

    def __init__(self, shape: synth.LayerShape, seed: int, tile_rows: int = 128,
                 zipf_s=None, device="cuda", experts=None, router_b=None,
                 out_dtype=lily.LILY_DTYPE_F32):
        self.shape = shape
        self.inp = synth.make_layer(shape, seed, device=device, zipf_s=zipf_s)
        if experts is not None:
            self.inp["experts"] = experts
        if router_b is not None:
            self.inp["router_b"] = router_b
        self.dims = lily.make_dims(shape.T, shape.d, shape.E, shape.k, shape.F, tile_rows,
                                   out_dtype=out_dtype)
        self.w = lily.LayerWeights(self.inp["router_w"], self.inp["router_b"], self.inp["experts"])
        self.r = lily.RoutingBuffers(self.dims, device)
        self.ws = lily.alloc_workspace(lily.lily_moe_workspace_bytes(self.dims), device)
        self.y = torch.empty(shape.T, shape.d, dtype=lily.out_torch_dtype(self.dims), device=device)
        self._np_experts = None

    @property
    def x(self):
        return self.inp["x"]

    def np_experts(self):
        if self._np_experts is None:
            self._np_experts = synth.experts_to_numpy(self.inp["experts"])
        return self._np_experts

    def forward(self):
        lily.lily_moe_forward(self.dims, self.x, self.w, self.r, self.y, self.ws)
        torch.cuda.synchronize()
        return self.y

    def decode(self):
        lily.lily_moe_decode(self.dims, self.x, self.w, self.r, self.y, self.ws)
        torch.cuda.synchronize()
        return self.y

    def status(self):
        return lily.lily_moe_status(self.ws)

    def oracle_route(self):
        return oracle.route(self.r.logits.cpu().numpy(), self.shape.k, self.dims.tile_rows)

    def oracle_rows(self, rows, ro=None):
        ro = ro or self.oracle_route()
        return oracle.moe_rows(synth.bf16_bits(self.x), self.np_experts(), ro["ids"], ro["gates"],
                               np.asarray(rows, np.int32))


def assert_routing_equal(gpu: dict, ro: dict, T: int, k: int):
    """Bit-exact routing given the same fp32 logits; gates within GATE_TOL."""
    assert np.array_equal(gpu["topk_ids"], ro["ids"]), "top-k ids differ"
    for name, ref in (("counts", ro["counts"]), ("offsets", ro["offsets"]), ("perm", ro["perm"]),
                      ("inv_perm", ro["inv"])):
        assert np.array_equal(gpu[name], ref), f"{name} differs"
    assert int(gpu["n_tiles"][0]) == ro["n_tiles"], "n_tiles differs"
    assert np.array_equal(gpu["block_map"], ro["block_map"]), "block map differs"
    g = gpu["topk_gates"].astype(np.float64)
    assert np.max(np.abs(g - ro["gates"])) <= GATE_TOL
    assert np.max(np.abs(g.sum(axis=1) - 1.0)) <= GATE_TOL
