"""The router weights' three-term bf16 split made once (lily_moe_router_split)
instead of on every call: the same logits and layer output, bit for bit, and
the split itself exact (hi + mid + lo == w in fp32)."""
import numpy as np
import pytest
import torch

import oracle
import w4_grouped_gemm_gb300 as lily
from w4_grouped_gemm_gb300 import synth

from gpu_util import Layer, assert_layer_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape,bm", [
    (synth.SHAPES["small"], 32),
    (synth.SHAPES["prefill512"], 64),
])
def test_presplit_router_gives_the_same_layer(oracle_lib, shape, bm):
    L = Layer(shape, seed=8800, tile_rows=bm)
    L.forward()
    torch.cuda.synchronize()
    logits0, y0 = L.r.logits.clone(), L.y.clone()
    L.w.split_router()
    L.forward()
    torch.cuda.synchronize()
    assert torch.equal(L.r.logits, logits0)
    assert torch.equal(L.y, y0)
    assert L.status() == 0
    # the layer still matches the oracle (sampled rows)
    sel = np.random.default_rng(3).choice(shape.T, min(shape.T, 24), replace=False)
    ro = oracle.route(L.r.logits.cpu().numpy(), shape.k, bm)
    ref = oracle.moe_rows(synth.bf16_bits(L.x), L.np_experts(), ro["ids"], ro["gates"],
                          sel.astype(np.int32))
    assert_layer_close(L.y.cpu().numpy()[sel], ref, "presplit router")


def test_router_split_is_exact():
    E, d = 256, 2048
    w = synth.make_router(E, d, 4242, "cuda")[0]
    split = torch.empty(lily.lib().lily_moe_router_split_bytes(E, d) // 2, dtype=torch.bfloat16,
                        device="cuda")
    lily.lily_moe_router_split(w, split)
    torch.cuda.synchronize()
    parts = split.view(3, E, d).float().double()
    wd = w.double()
    # each term is a bf16 value, and the three add up to w exactly
    assert torch.equal(parts.sum(0), wd)
    # the terms are the successive bf16 roundings of the remainders
    hi = w.bfloat16()
    assert torch.equal(split.view(3, E, d)[0], hi)
