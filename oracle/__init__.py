"""FP64 CPU oracle for the W4 MoE expert layer -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library and its Python
binding) never loads it, and the oracle shares no code with that path: it is a
separate C++ translation unit (``lily_oracle.cpp``) compiled with the host C++
compiler and loaded here through ctypes.

Every function takes and returns numpy arrays.  bf16 tensors travel as their raw
``uint16`` bit patterns.  See ``lily_oracle.cpp`` for the definitions and the
passages of the Lily pages each one follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "lily_oracle.cpp"
_LIB = _HERE / "liblily_oracle.so"
_lib = None


def build(force: bool = False) -> Path:
    """Compile the oracle with g++ (plain -O2, no fast-math: IEEE double)."""
    if force or not _LIB.exists() or _LIB.stat().st_mtime < _SRC.stat().st_mtime:
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", str(_SRC), "-o", str(_LIB) + ".tmp"]
        subprocess.run(cmd, check=True)
        os.replace(str(_LIB) + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(str(_LIB))
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.orc_dequant.argtypes = [I, I, P, P, P, P]
        lib.orc_router_logits.argtypes = [I, I, I, P, P, P, P, P]
        lib.orc_block_map_cap.argtypes = [I, I, I, I]
        lib.orc_route.argtypes = [I, I, I, I, P, P, P, P, P, P, P, P, I, P, P]
        lib.orc_moe_rows.argtypes = [I, I, I, I, I, P] + [P] * 9 + [P, P, I, P, P]
        lib.orc_moe_layer.argtypes = [I, I, I, I, I, I, P, P, P] + [P] * 9 + [P, P, P]
        lib.orc_rmsnorm.argtypes = [I, I, P, ctypes.c_double, P]
        for f in ("orc_dequant", "orc_router_logits", "orc_block_map_cap", "orc_route",
                  "orc_moe_rows", "orc_moe_layer", "orc_rmsnorm"):
            getattr(lib, f).restype = I
        _lib = lib
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


def dequant(q, s, b):
    """w = s*q + b per 64-element group, in float64.  q: uint8 [R][C/2]."""
    q, qp = _c(q, np.uint8)
    s, sp = _c(s, np.uint16)
    b, bp = _c(b, np.uint16)
    R, C = q.shape[0], q.shape[1] * 2
    w = np.empty((R, C), np.float64)
    _check(_load().orc_dequant(R, C, qp, sp, bp, _ptr(w)), "dequant")
    return w


def router_logits(x_bits, wr, br=None):
    """(logits[T][E], abs_sum[T][E]) in float64."""
    x, xp = _c(x_bits, np.uint16)
    wr, wp = _c(wr, np.float32)
    T, d = x.shape
    E = wr.shape[0]
    brp = None
    if br is not None:
        br, brp = _c(br, np.float32)
    L = np.empty((T, E), np.float64)
    A = np.empty((T, E), np.float64)
    _check(_load().orc_router_logits(T, d, E, xp, wp, brp, _ptr(L), _ptr(A)), "router_logits")
    return L, A


def block_map_cap(T, E, k, BM):
    return int(_load().orc_block_map_cap(T, E, k, BM))


def route(logits_f32, k, BM):
    """Routing from fp32 logits [T][E].  Returns a dict of numpy arrays."""
    L, Lp = _c(logits_f32, np.float32)
    T, E = L.shape
    P = T * k
    cap = block_map_cap(T, E, k, BM)
    out = dict(
        ids=np.empty((T, k), np.int32), gates=np.empty((T, k), np.float64),
        counts=np.empty(E, np.int32), offsets=np.empty(E + 1, np.int32),
        perm=np.empty(P, np.int32), inv=np.empty(P, np.int32),
        block_map=np.empty((cap, 2), np.int32),
    )
    nt = np.zeros(1, np.int32)
    nn = np.zeros(1, np.int32)
    rc = _load().orc_route(T, E, k, BM, Lp, _ptr(out["ids"]), _ptr(out["gates"]),
                           _ptr(out["counts"]), _ptr(out["offsets"]), _ptr(out["perm"]),
                           _ptr(out["inv"]), _ptr(out["block_map"]), cap, _ptr(nt), _ptr(nn))
    _check(rc, "route")
    out["n_tiles"] = int(nt[0])
    out["n_nan"] = int(nn[0])
    return out


_WNAMES = ("gate_q", "gate_s", "gate_b", "up_q", "up_s", "up_b", "down_q", "down_s", "down_b")


def _weights(w):
    arrs, ptrs = [], []
    for n in _WNAMES:
        a, p = _c(w[n], np.uint8 if n.endswith("_q") else np.uint16)
        arrs.append(a)
        ptrs.append(p)
    return arrs, ptrs


def moe_rows(x_bits, w, ids, gates, rows):
    """Layer output (float64 [len(rows)][d]) for the given token rows.

    ``w`` maps gate_q/gate_s/gate_b/up_q/up_s/up_b/down_q/down_s/down_b to numpy
    arrays holding E+1 experts (the last is the shared expert)."""
    x, xp = _c(x_bits, np.uint16)
    T, d = x.shape
    ids, ip = _c(ids, np.int32)
    gates, gp = _c(gates, np.float64)
    rows, rp = _c(rows, np.int32)
    k = ids.shape[1]
    E = w["gate_q"].shape[0] - 1
    F = w["gate_q"].shape[1]
    arrs, ptrs = _weights(w)
    y = np.empty((rows.shape[0], d), np.float64)
    rc = _load().orc_moe_rows(T, d, E, k, F, xp, *ptrs, ip, gp, len(rows), rp, _ptr(y))
    _check(rc, "moe_rows")
    return y


def moe_layer(x_bits, wr, br, w, k, BM):
    """The whole layer from scratch (double logits rounded to fp32 for routing)."""
    x, xp = _c(x_bits, np.uint16)
    T, d = x.shape
    wr, wp = _c(wr, np.float32)
    brp = None
    if br is not None:
        br, brp = _c(br, np.float32)
    E = w["gate_q"].shape[0] - 1
    F = w["gate_q"].shape[1]
    arrs, ptrs = _weights(w)
    ids = np.empty((T, k), np.int32)
    gates = np.empty((T, k), np.float64)
    y = np.empty((T, d), np.float64)
    rc = _load().orc_moe_layer(T, d, E, k, F, BM, xp, wp, brp, *ptrs, _ptr(ids), _ptr(gates), _ptr(y))
    _check(rc, "moe_layer")
    return y, ids, gates


def rmsnorm(x_f32, eps=1e-6):
    x, xp = _c(x_f32, np.float32)
    T, d = x.shape
    out = np.empty((T, d), np.float64)
    _check(_load().orc_rmsnorm(T, d, xp, float(eps), _ptr(out)), "rmsnorm")
    return out
