"""Pins for the FP64 CPU oracle (no GPU).

Each test ties the oracle to something other than itself: hand-worked values
(tests/golden), brute force on tiny inputs, library routines (numpy/torch/scipy
float64), closed forms of the layer, and invariants of the routing stages.
"""
import itertools
import math
from pathlib import Path

import numpy as np
import pytest
import torch

GOLDEN = Path(__file__).resolve().parent / "golden"


def _read_fixture(name):
    out = {}
    for line in (GOLDEN / name).read_text().splitlines():
        if not line.strip() or line.startswith("#"):
            continue
        key, *vals = line.split()
        out[key] = vals
    return out


def _f32_to_bf16_bits(a):
    """Round-to-nearest-even fp32 -> bf16 bit patterns (numpy)."""
    a = np.ascontiguousarray(a, np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    return r


def _bf16_bits_to_f64(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _rand_experts(rng, E, d, F, scale_lo=0.001, scale_hi=0.01):
    def mat(n, rows, cols):
        q = rng.integers(0, 256, size=(n, rows, cols // 2), dtype=np.uint8)
        s = _f32_to_bf16_bits(rng.uniform(scale_lo, scale_hi, size=(n, rows, cols // 64)))
        b = _f32_to_bf16_bits(rng.uniform(-0.08, 0.0, size=(n, rows, cols // 64)))
        return q, s, b
    gq, gs, gb = mat(E + 1, F, d)
    uq, us, ub = mat(E + 1, F, d)
    dq, ds, db = mat(E + 1, d, F)
    return dict(gate_q=gq, gate_s=gs, gate_b=gb, up_q=uq, up_s=us, up_b=ub,
                down_q=dq, down_s=ds, down_b=db)


def _rand_x(rng, T, d):
    return _f32_to_bf16_bits(rng.standard_normal((T, d)).astype(np.float32))


# ----------------------------------------------------------------- dequant

def test_dequant_golden_nibble_order(oracle):
    fx = _read_fixture("dequant_nibble_order.txt")
    C = int(fx["C"][0])
    q = np.zeros((1, C // 2), np.uint8)
    for item in fx["bytes"]:
        pos, val = item.split(":")
        q[0, int(pos)] = int(val, 16)
    s = np.array([[int(v, 16) for v in fx["scale"]]], np.uint16)
    b = np.array([[int(v, 16) for v in fx["bias"]]], np.uint16)
    w = oracle.dequant(q, s, b)
    for item in fx["expect"]:
        pos, val = item.split(":")
        assert w[0, int(pos)] == float(val), (pos, w[0, int(pos)], val)


def test_dequant_special_cases(oracle):
    rng = np.random.default_rng(1)
    R, C = 5, 256
    s = _f32_to_bf16_bits(rng.uniform(0.001, 0.01, (R, C // 64)))
    b = _f32_to_bf16_bits(rng.uniform(-0.08, 0.0, (R, C // 64)))
    sf, bf = _bf16_bits_to_f64(s), _bf16_bits_to_f64(b)
    # q = 0  =>  w = bias
    w = oracle.dequant(np.zeros((R, C // 2), np.uint8), s, b)
    assert np.array_equal(w, np.repeat(bf, 64, axis=1))
    # scale = 0  =>  w = bias (a per-group constant) whatever q is
    q = rng.integers(0, 256, (R, C // 2), dtype=np.uint8)
    w = oracle.dequant(q, np.zeros_like(s), b)
    assert np.array_equal(w, np.repeat(bf, 64, axis=1))
    # q = 15, bias = 0  =>  w = 15 * scale
    w = oracle.dequant(np.full((R, C // 2), 0xFF, np.uint8), s, np.zeros_like(b))
    assert np.array_equal(w, 15.0 * np.repeat(sf, 64, axis=1))


def test_dequant_group_boundary(oracle):
    """Elements 0..63 use group 0's scale/bias and 64..127 group 1's."""
    rng = np.random.default_rng(2)
    q = rng.integers(0, 256, (1, 64), dtype=np.uint8)
    s = _f32_to_bf16_bits(np.array([[0.5, 0.25]], np.float32))
    b = _f32_to_bf16_bits(np.array([[0.0, 0.0]], np.float32))
    w1 = oracle.dequant(q, s, b)
    s2 = _f32_to_bf16_bits(np.array([[0.5, 2.0]], np.float32))
    w2 = oracle.dequant(q, s2, b)
    assert np.array_equal(w1[0, :64], w2[0, :64])
    assert np.array_equal(w2[0, 64:], 8.0 * w1[0, 64:])


# ----------------------------------------------------------------- routing

def test_route_golden(oracle):
    fx = _read_fixture("routing_small.txt")
    T, E, k, BM = (int(fx[n][0]) for n in ("T", "E", "k", "BM"))
    L = np.array([float(v) for v in fx["logits"]], np.float32).reshape(T, E)
    r = oracle.route(L, k, BM)
    assert r["ids"].ravel().tolist() == [int(v) for v in fx["ids"]]
    np.testing.assert_allclose(r["gates"].ravel(), [float(v) for v in fx["gates"]], rtol=0, atol=1e-15)
    for name in ("counts", "offsets", "perm", "inv"):
        assert r[name].tolist() == [int(v) for v in fx[name]], name
    assert r["n_tiles"] == int(fx["n_tiles"][0])
    assert r["block_map"].ravel().tolist() == [int(v) for v in fx["block_map"]]


def _brute_topk(L, k):
    """Slot of each expert = number of experts ranking before it (counting)."""
    T, E = L.shape
    ids = np.full((T, k), -1, np.int64)
    for t in range(T):
        for e in range(E):
            rank = sum(1 for f in range(E) if L[t, f] > L[t, e] or (L[t, f] == L[t, e] and f < e))
            if rank < k:
                ids[t, rank] = e
    return ids


@pytest.mark.parametrize("seed", range(12))
def test_route_bruteforce_tiny(oracle, seed):
    rng = np.random.default_rng(100 + seed)
    T = int(rng.integers(1, 5))
    E = int(rng.integers(2, 9))
    k = int(rng.integers(1, min(E, 3) + 1))
    BM = int(rng.integers(1, 4))
    L = rng.integers(-2, 3, size=(T, E)).astype(np.float32)   # many ties
    r = oracle.route(L, k, BM)
    assert np.array_equal(r["ids"], _brute_topk(L, k))
    P = T * k
    flat = r["ids"].ravel()
    # histogram by exhaustive counting
    assert r["counts"].tolist() == [int(np.sum(flat == e)) for e in range(E)]
    # perm = pairs stably sorted by expert (library stable sort)
    ref = sorted(range(P), key=lambda p: (flat[p], p))
    assert r["perm"].tolist() == ref
    # block map: every (expert, row-range) tiling enumerated the slow way
    tiles = []
    for e in range(E):
        rows = [pos for pos in range(P) if flat[ref[pos]] == e]
        for i in range(0, len(rows), BM):
            tiles.append((e, rows[i]))
    assert r["n_tiles"] == len(tiles)
    assert [tuple(t) for t in r["block_map"][: len(tiles)].tolist()] == tiles
    assert np.all(r["block_map"][len(tiles):] == -1)


def _check_routing_invariants(r, T, E, k, BM):
    P = T * k
    ids, counts, offsets, perm, inv = r["ids"], r["counts"], r["offsets"], r["perm"], r["inv"]
    assert counts.sum() == P
    assert offsets[0] == 0 and offsets[E] == P
    assert np.all(np.diff(offsets) == counts) and np.all(np.diff(offsets) >= 0)
    assert sorted(perm.tolist()) == list(range(P))            # a permutation
    assert np.array_equal(inv[perm], np.arange(P))            # inv o perm = id
    experts_along = ids.ravel()[perm]
    assert np.all(np.diff(experts_along) >= 0)                # expert-contiguous
    for e in range(E):                                        # stable in pair index
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)
        assert np.all(ids.ravel()[seg] == e)
    for t in range(T):                                        # k distinct experts
        assert len(set(ids[t].tolist())) == k
    np.testing.assert_allclose(r["gates"].sum(axis=1), 1.0, rtol=0, atol=1e-12)
    # tiles cover [0, P) once, never cross an expert boundary, ordered
    nt = r["n_tiles"]
    bm = r["block_map"]
    covered = np.zeros(P, np.int32)
    last = (-1, -1)
    for i in range(nt):
        e, rb = int(bm[i, 0]), int(bm[i, 1])
        re = min(rb + BM, int(offsets[e + 1]))
        assert offsets[e] <= rb < re <= offsets[e + 1]
        assert (e, rb) > last
        last = (e, rb)
        covered[rb:re] += 1
    assert np.all(covered == 1)
    assert np.all(bm[nt:] == -1)
    assert nt == sum(-(-int(c) // BM) for c in counts)


@pytest.mark.parametrize("T,E,k,BM", [(64, 32, 4, 8), (37, 16, 3, 5), (1, 256, 8, 32), (200, 256, 8, 32)])
def test_route_invariants(oracle, T, E, k, BM):
    rng = np.random.default_rng(T * 1000 + E)
    L = rng.standard_normal((T, E)).astype(np.float32)
    r = oracle.route(L, k, BM)
    _check_routing_invariants(r, T, E, k, BM)
    assert r["n_nan"] == 0


def test_route_skewed_and_single_expert(oracle):
    """All tokens prefer one expert (bias), and E == k (every expert chosen)."""
    rng = np.random.default_rng(5)
    T, E, k, BM = 50, 16, 2, 8
    L = rng.standard_normal((T, E)).astype(np.float32)
    L[:, 7] += 100.0
    r = oracle.route(L, k, BM)
    _check_routing_invariants(r, T, E, k, BM)
    assert np.all(r["ids"][:, 0] == 7) and r["counts"][7] == T
    r = oracle.route(L[:, :4], 4, 3)
    _check_routing_invariants(r, T, 4, 4, 3)
    assert all(sorted(row) == [0, 1, 2, 3] for row in r["ids"].tolist())


def test_gates_are_renormalised_softmax(oracle):
    """Gates = full softmax (scipy) renormalised over the kept experts."""
    from scipy.special import softmax
    rng = np.random.default_rng(7)
    T, E, k = 20, 64, 8
    L = (3 * rng.standard_normal((T, E))).astype(np.float32)
    r = oracle.route(L, k, 16)
    full = softmax(L.astype(np.float64), axis=1)
    sel = np.take_along_axis(full, r["ids"].astype(np.int64), axis=1)
    np.testing.assert_allclose(r["gates"], sel / sel.sum(axis=1, keepdims=True), rtol=1e-13, atol=0)
    # order within a token: gates non-increasing along the slots
    assert np.all(np.diff(r["gates"], axis=1) <= 1e-15)


def test_route_nan_and_inf(oracle):
    L = np.array([[np.nan, 1.0, 2.0, np.nan],
                  [np.nan, np.nan, np.nan, 0.5],
                  [-np.inf, -np.inf, -np.inf, -np.inf],
                  [np.inf, 1.0, np.inf, 0.0]], np.float32)
    r = oracle.route(L, 2, 4)
    assert r["n_nan"] == 5
    assert r["ids"][0].tolist() == [2, 1]          # NaN ranks below every number
    assert r["ids"][1].tolist() == [3, 0]          # then NaNs by id
    assert r["ids"][2].tolist() == [0, 1]          # all -inf: ties by id
    np.testing.assert_array_equal(r["gates"][2], [0.5, 0.5])
    assert r["ids"][3].tolist() == [0, 2]
    np.testing.assert_array_equal(r["gates"][3], [0.5, 0.5])


# ----------------------------------------------------------------- router

def test_router_logits_vs_numpy(oracle):
    rng = np.random.default_rng(9)
    T, d, E = 7, 192, 12
    x = _rand_x(rng, T, d)
    wr = (0.02 * rng.standard_normal((E, d))).astype(np.float32)
    br = rng.standard_normal(E).astype(np.float32)
    L, A = oracle.router_logits(x, wr, br)
    xf = _bf16_bits_to_f64(x)
    ref = xf @ wr.astype(np.float64).T + br.astype(np.float64)
    np.testing.assert_allclose(L, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(A, np.abs(xf) @ np.abs(wr.astype(np.float64)).T, rtol=1e-12)
    L0, _ = oracle.router_logits(x, wr, None)
    np.testing.assert_allclose(L0, xf @ wr.astype(np.float64).T, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------- expert FFN / layer

def _torch_ffn(oracle, w, e, x64):
    """SwiGLU FFN of expert e in torch float64 on explicitly dequantised W."""
    Wg = torch.from_numpy(oracle.dequant(w["gate_q"][e], w["gate_s"][e], w["gate_b"][e]))
    Wu = torch.from_numpy(oracle.dequant(w["up_q"][e], w["up_s"][e], w["up_b"][e]))
    Wd = torch.from_numpy(oracle.dequant(w["down_q"][e], w["down_s"][e], w["down_b"][e]))
    x = torch.from_numpy(x64)
    h = torch.nn.functional.silu(x @ Wg.T) * (x @ Wu.T)
    return (h @ Wd.T).numpy()


def test_layer_vs_torch_float64(oracle):
    """y = sum_j g_j FFN_{e_j}(x) + FFN_shared(x), checked with torch matmul/silu."""
    rng = np.random.default_rng(11)
    T, d, E, k, F = 6, 128, 5, 2, 192
    w = _rand_experts(rng, E, d, F)
    x = _rand_x(rng, T, d)
    L = rng.standard_normal((T, E)).astype(np.float32)
    r = oracle.route(L, k, 4)
    y = oracle.moe_rows(x, w, r["ids"], r["gates"], np.arange(T))
    x64 = _bf16_bits_to_f64(x)
    ref = _torch_ffn(oracle, w, E, x64)
    for t in range(T):
        for j in range(k):
            ref[t] += r["gates"][t, j] * _torch_ffn(oracle, w, int(r["ids"][t, j]), x64[t:t + 1])[0]
    np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-12)
    # a row subset gives the same rows
    ys = oracle.moe_rows(x, w, r["ids"], r["gates"], np.array([4, 1]))
    np.testing.assert_array_equal(ys, y[[4, 1]])


def test_layer_closed_form_identical_experts(oracle):
    """All routed experts and the shared expert identical => y = 2 * FFN(x)."""
    rng = np.random.default_rng(12)
    T, d, E, k, F = 9, 64, 6, 3, 128
    w1 = _rand_experts(rng, 0, d, F)                 # one expert
    w = {n: np.repeat(a, E + 1, axis=0) for n, a in w1.items()}
    x = _rand_x(rng, T, d)
    L = rng.standard_normal((T, E)).astype(np.float32)
    r = oracle.route(L, k, 4)
    y = oracle.moe_rows(x, w, r["ids"], r["gates"], np.arange(T))
    ffn = _torch_ffn(oracle, w1, 0, _bf16_bits_to_f64(x))
    np.testing.assert_allclose(y, 2.0 * ffn, rtol=1e-12, atol=1e-13)
    # and with E == k every expert is used by every token
    r = oracle.route(L[:, :k], k, 4)
    assert all(sorted(row) == list(range(k)) for row in r["ids"].tolist())


def test_layer_zero_gate_projection(oracle):
    """Gate-projection weights all zero => silu(0) = 0 => y = 0 exactly."""
    rng = np.random.default_rng(13)
    T, d, E, k, F = 4, 64, 3, 2, 64
    w = _rand_experts(rng, E, d, F)
    w["gate_s"][:] = 0
    w["gate_b"][:] = 0
    x = _rand_x(rng, T, d)
    r = oracle.route(rng.standard_normal((T, E)).astype(np.float32), k, 2)
    y = oracle.moe_rows(x, w, r["ids"], r["gates"], np.arange(T))
    assert np.all(y == 0.0)


def test_moe_layer_from_scratch_matches_parts(oracle):
    rng = np.random.default_rng(14)
    T, d, E, k, F = 5, 64, 4, 2, 64
    w = _rand_experts(rng, E, d, F)
    x = _rand_x(rng, T, d)
    wr = (0.02 * rng.standard_normal((E, d))).astype(np.float32)
    y, ids, gates = oracle.moe_layer(x, wr, None, w, k, 2)
    L, _ = oracle.router_logits(x, wr, None)
    r = oracle.route(L.astype(np.float32), k, 2)
    assert np.array_equal(ids, r["ids"])
    np.testing.assert_array_equal(y, oracle.moe_rows(x, w, r["ids"], r["gates"], np.arange(T)))


# ----------------------------------------------------------------- rmsnorm

def test_rmsnorm(oracle):
    c = np.full((1, 64), -3.0, np.float32)
    out = oracle.rmsnorm(c, eps=1e-6)
    np.testing.assert_allclose(out, -3.0 / math.sqrt(9.0 + 1e-6), rtol=1e-15)
    rng = np.random.default_rng(15)
    x = rng.standard_normal((3, 96)).astype(np.float32) * 5
    out = oracle.rmsnorm(x, eps=1e-6)
    x64 = x.astype(np.float64)
    ref = x64 / np.sqrt((x64 ** 2).mean(axis=1, keepdims=True) + 1e-6)
    np.testing.assert_allclose(out, ref, rtol=1e-13)
