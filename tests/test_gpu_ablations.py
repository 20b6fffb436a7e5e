"""The benchmark's two ablation arms compute the same layer: host-synced
routing (block map built on the host) and weights dequantised to fp16 in HBM
followed by batched cuBLAS GEMMs.  Each arm's output is checked against the
FP64 oracle (routed from the GPU's fp32 logits), so the ablation timings
compare implementations of one and the same layer."""
import numpy as np
import pytest
import torch

import bench
import oracle
import w4_grouped_gemm_gb300 as lily
from w4_grouped_gemm_gb300 import synth

from gpu_util import assert_layer_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape,bm,rows", [
    (synth.SHAPES["small"], 32, None),
    (synth.SHAPES["prefill512"], 64, 24),
])
@pytest.mark.parametrize("name", ["host_routing", "dequant_hbm"])
def test_ablation_matches_oracle(oracle_lib, shape, bm, rows, name):
    ab = bench.Ablation(lily, synth, shape, bm, seed=7700, dev=torch.device("cuda"))
    ab.run(name)
    torch.cuda.synchronize()
    T = shape.T
    sel = np.arange(T) if rows is None else np.random.default_rng(7).choice(T, rows, replace=False)
    ro = oracle.route(ab.r.logits.cpu().numpy(), shape.k, bm)
    ref = oracle.moe_rows(synth.bf16_bits(ab.x), synth.experts_to_numpy(ab.inp["experts"]),
                          ro["ids"], ro["gates"], sel.astype(np.int32))
    got = ab.y.cpu().numpy()[sel]
    assert_layer_close(got, ref, f"ablation {name}")
