"""ctypes binding of liblily_moe.so (the C ABI in include/lily_moe.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  torch is used for device memory and streams.  The binding refuses to
work without the compiled library -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import operator
from dataclasses import dataclass
from pathlib import Path

import torch

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "liblily_moe.so"

LILY_OK = 0
LILY_ERR_INVALID_ARG = -1
LILY_ERR_UNSUPPORTED_SHAPE = -2
LILY_ERR_MISALIGNED = -3
LILY_ERR_WORKSPACE_TOO_SMALL = -4
LILY_ERR_ARCH = -5
LILY_ERR_CUDA = -6
LILY_ERR_DEVICE = -7
LILY_STATUS_NAN_LOGIT = 0x1
LILY_STATUS_TIMEOUT = 0x2
LILY_STATUS_BAD_TILE = 0x4
LILY_STATUS_F16_RANGE = 0x8
LILY_KERNEL_KINDS = 16

# Every symbol include/lily_moe.h declares.
EXPORTS = (
    "lily_moe_workspace_bytes", "lily_moe_block_map_cap", "lily_moe_check_dims",
    "lily_moe_route", "lily_moe_forward", "lily_moe_experts", "lily_moe_decode",
    "lily_moe_decode_static",
    "lily_moe_forward_host", "lily_moe_forward_host_async", "lily_moe_host_graphs",
    "lily_moe_rmsnorm", "lily_moe_stack_prefill", "lily_moe_stack_decode",
    "lily_moe_router_split_bytes", "lily_moe_router_split",
    "lily_moe_stack_workspace_bytes",
    "lily_moe_status", "lily_moe_set_route_wait_ns", "lily_moe_strerror", "lily_moe_profile_enable", "lily_moe_profile_read",
    "lily_moe_kernel_name", "lily_moe_version",
)


class LilyError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {strerror(code)} ({code})")
        self.code = code


LILY_DTYPE_BF16 = 0
LILY_DTYPE_F32 = 1


class Dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d_model", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("d_ff", ctypes.c_int32), ("group", ctypes.c_int32),
                ("tile_rows", ctypes.c_int32), ("out_dtype", ctypes.c_int32)]


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "router_w", "router_bias", "gate_q", "gate_s", "gate_b", "up_q", "up_s", "up_b",
        "down_q", "down_s", "down_b", "router_w_split")]


class Routing(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "logits", "topk_ids", "topk_gates", "counts", "offsets", "perm", "inv_perm",
        "block_map", "n_tiles")]


_lib = None


def lib():
    """The loaded library; raises if it was not built (no fallback)."""
    global _lib
    if _lib is None:
        if not LIB_PATH.exists():
            raise RuntimeError(f"{LIB_PATH.name} is not built: run __graft_entry__.build() "
                               "(nvcc, sm_103a) first; this package has no CPU fallback")
        L = ctypes.CDLL(str(LIB_PATH))
        P, I, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        DP, WP, RP = ctypes.POINTER(Dims), ctypes.POINTER(Weights), ctypes.POINTER(Routing)
        sig = {
            "lily_moe_workspace_bytes": (SZ, [DP]),
            "lily_moe_stack_workspace_bytes": (SZ, [DP]),
            "lily_moe_block_map_cap": (ctypes.c_int64, [DP]),
            "lily_moe_check_dims": (I, [DP]),
            "lily_moe_route": (I, [DP, P, P, WP, RP, P, SZ, P]),
            "lily_moe_forward": (I, [DP, P, WP, RP, P, P, SZ, P]),
            "lily_moe_experts": (I, [DP, P, WP, RP, P, P, SZ, P]),
            "lily_moe_decode": (I, [DP, P, WP, RP, P, P, SZ, P]),
            "lily_moe_decode_static": (I, [DP, P, WP, RP, P, P]),
            "lily_moe_forward_host": (I, [DP, P, P, WP, RP, P, P, P, SZ, P]),
            "lily_moe_forward_host_async": (I, [DP, P, P, WP, RP, P, P, P, SZ, P]),
            "lily_moe_host_graphs": (I, [I]),
            "lily_moe_rmsnorm": (I, [ctypes.c_int32, ctypes.c_int32, P, ctypes.c_float, P, P]),
            "lily_moe_router_split_bytes": (SZ, [ctypes.c_int32, ctypes.c_int32]),
            "lily_moe_router_split": (I, [P, ctypes.c_int32, ctypes.c_int32, P, P]),
            "lily_moe_stack_prefill": (I, [DP, ctypes.c_int32, ctypes.c_int32, WP, P,
                                           ctypes.c_float, P, P, P, SZ, P]),
            "lily_moe_stack_decode": (I, [DP, ctypes.c_int32, WP, P, ctypes.c_float, P, P, P,
                                          SZ, P]),
            "lily_moe_status": (I, [P, P]),
            "lily_moe_set_route_wait_ns": (ctypes.c_uint64, [ctypes.c_uint64]),
            "lily_moe_strerror": (ctypes.c_char_p, [I]),
            "lily_moe_profile_enable": (I, [I]),
            "lily_moe_profile_read": (I, [P, P]),
            "lily_moe_kernel_name": (ctypes.c_char_p, [I]),
            "lily_moe_version": (ctypes.c_char_p, []),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def strerror(code: int) -> str:
    return lib().lily_moe_strerror(int(code)).decode()


def _check(rc: int, what: str):
    if rc != LILY_OK:
        raise LilyError(rc, what)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream):
    if stream is None:
        if _raw_stream is not None:  # the current stream's handle, no Stream object
            return _raw_stream(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_dims(T, d, E, k, F, tile_rows=128, group=64, out_dtype=LILY_DTYPE_F32) -> Dims:
    return Dims(T, d, E, k, F, group, tile_rows, out_dtype)


def out_torch_dtype(dims: Dims):
    return torch.float32 if dims.out_dtype == LILY_DTYPE_F32 else torch.bfloat16


def lily_moe_check_dims(dims: Dims) -> int:
    return lib().lily_moe_check_dims(ctypes.byref(dims))


def lily_moe_workspace_bytes(dims: Dims) -> int:
    return int(lib().lily_moe_workspace_bytes(ctypes.byref(dims)))


def lily_moe_stack_workspace_bytes(dims: Dims) -> int:
    return int(lib().lily_moe_stack_workspace_bytes(ctypes.byref(dims)))


def lily_moe_block_map_cap(dims: Dims) -> int:
    return int(lib().lily_moe_block_map_cap(ctypes.byref(dims)))


def _cached_view(owner, refs: tuple, struct):
    """ctypes struct of the tensors `refs`, rebuilt only when one of them is
    replaced by another object (a call then costs no data_ptr() lookups)."""
    hit = owner.__dict__.get("_cview")
    if hit is not None and all(map(operator.is_, hit[0], refs)):
        return hit[1]
    view = struct(*(_ptr(t) for t in refs))
    owner.__dict__["_cview"] = (refs, view)
    return view


@dataclass
class LayerWeights:
    """torch tensors of one layer; .c is the ctypes view (keeps the tensors alive).
    router_split: the router weights' three-term bf16 split made once by
    lily_moe_router_split (or None: the library splits on every call)."""
    router_w: torch.Tensor
    router_b: torch.Tensor | None
    experts: dict
    router_split: torch.Tensor | None = None

    @property
    def c(self) -> Weights:
        e = self.experts
        refs = (self.router_w, self.router_b, e["gate_q"], e["gate_s"], e["gate_b"], e["up_q"],
                e["up_s"], e["up_b"], e["down_q"], e["down_s"], e["down_b"], self.router_split)
        return _cached_view(self, refs, Weights)

    def split_router(self, stream=None) -> "LayerWeights":
        """Make the router weights' split once (lily_moe_router_split); later
        calls with these weights skip the per-call split."""
        E, d = self.router_w.shape
        n = lib().lily_moe_router_split_bytes(E, d)
        buf = torch.empty(n // 2, dtype=torch.bfloat16, device=self.router_w.device)
        lily_moe_router_split(self.router_w, buf, stream)
        self.router_split = buf
        return self


class RoutingBuffers:
    """Caller-owned routing outputs (device tensors) for one dims."""

    def __init__(self, dims: Dims, device="cuda"):
        T, E, k = dims.T, dims.n_experts, dims.top_k
        P = T * k
        cap = lily_moe_block_map_cap(dims)
        i32 = dict(dtype=torch.int32, device=device)
        self.logits = torch.empty(T, E, dtype=torch.float32, device=device)
        self.topk_ids = torch.empty(T, k, **i32)
        self.topk_gates = torch.empty(T, k, dtype=torch.float32, device=device)
        self.counts = torch.empty(E, **i32)
        self.offsets = torch.empty(E + 1, **i32)
        self.perm = torch.empty(P, **i32)
        self.inv_perm = torch.empty(P, **i32)
        self.block_map = torch.empty(cap, 2, **i32)
        self.n_tiles = torch.empty(1, **i32)

    @property
    def c(self) -> Routing:
        return _cached_view(self, tuple(getattr(self, n) for n, _ in Routing._fields_), Routing)

    def host(self) -> dict:
        return {n: getattr(self, n).cpu().numpy() for n, _ in Routing._fields_}


def alloc_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """Zero-filled device workspace (the library never allocates)."""
    return torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=device)


def lily_moe_route(dims, x, logits_in, weights: LayerWeights | None, routing: RoutingBuffers,
                   ws: torch.Tensor, stream=None):
    wc = weights.c if weights is not None else None
    rc = lib().lily_moe_route(ctypes.byref(dims), _ptr(x), _ptr(logits_in),
                              ctypes.byref(wc) if wc is not None else None,
                              ctypes.byref(routing.c), _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "lily_moe_route")


def lily_moe_forward(dims, x, weights: LayerWeights, routing: RoutingBuffers, y, ws, stream=None):
    rc = lib().lily_moe_forward(ctypes.byref(dims), _ptr(x), ctypes.byref(weights.c),
                                ctypes.byref(routing.c), _ptr(y), _ptr(ws), ws.numel(),
                                _stream(stream))
    _check(rc, "lily_moe_forward")


def lily_moe_experts(dims, x, weights: LayerWeights, routing: RoutingBuffers, y, ws, stream=None):
    """The expert GEMMs alone, from routing already in `routing`."""
    rc = lib().lily_moe_experts(ctypes.byref(dims), _ptr(x), ctypes.byref(weights.c),
                                ctypes.byref(routing.c), _ptr(y), _ptr(ws), ws.numel(),
                                _stream(stream))
    _check(rc, "lily_moe_experts")


def lily_moe_decode(dims, x, weights: LayerWeights, routing: RoutingBuffers, y, ws, stream=None):
    rc = lib().lily_moe_decode(ctypes.byref(dims), _ptr(x), ctypes.byref(weights.c),
                               ctypes.byref(routing.c), _ptr(y), _ptr(ws), ws.numel(),
                               _stream(stream))
    _check(rc, "lily_moe_decode")


def lily_moe_forward_host(dims, x_host, x_dev, weights: LayerWeights, routing: RoutingBuffers,
                          y_dev, y_host, ws, stream=None):
    rc = lib().lily_moe_forward_host(ctypes.byref(dims), _ptr(x_host), _ptr(x_dev),
                                     ctypes.byref(weights.c), ctypes.byref(routing.c),
                                     _ptr(y_dev), _ptr(y_host), _ptr(ws), ws.numel(),
                                     _stream(stream))
    _check(rc, "lily_moe_forward_host")


def lily_moe_forward_host_async(dims, x_host, x_dev, weights: LayerWeights,
                                routing: RoutingBuffers, y_dev, y_host, ws, stream=None):
    """lily_moe_forward_host without the final wait (see the header): the
    result is in y_host once `stream` has been synchronised."""
    rc = lib().lily_moe_forward_host_async(ctypes.byref(dims), _ptr(x_host), _ptr(x_dev),
                                           ctypes.byref(weights.c), ctypes.byref(routing.c),
                                           _ptr(y_dev), _ptr(y_host), _ptr(ws), ws.numel(),
                                           _stream(stream))
    _check(rc, "lily_moe_forward_host_async")


def lily_moe_host_graphs(enable: bool) -> bool:
    """Turn the end-to-end call's graph cache on or off (dropping cached
    graphs); returns the previous setting."""
    return bool(lib().lily_moe_host_graphs(1 if enable else 0))


def lily_moe_router_split(router_w, split, stream=None):
    E, d = router_w.shape
    _check(lib().lily_moe_router_split(_ptr(router_w), E, d, _ptr(split), _stream(stream)),
           "lily_moe_router_split")


def lily_moe_rmsnorm(x, out, eps=1e-6, stream=None):
    T, d = x.shape
    _check(lib().lily_moe_rmsnorm(T, d, _ptr(x), eps, _ptr(out), _stream(stream)),
           "lily_moe_rmsnorm")


def lily_moe_stack_prefill(dims, x, layers: list, eps=1e-6, layer_inputs=None,
                           layer_logits=None, ws=None, stream=None):
    arr = (Weights * len(layers))(*[l.c for l in layers])
    T_total = x.shape[0]
    rc = lib().lily_moe_stack_prefill(ctypes.byref(dims), T_total, len(layers), arr, _ptr(x), eps,
                                      _ptr(layer_inputs), _ptr(layer_logits), _ptr(ws),
                                      ws.numel(), _stream(stream))
    _check(rc, "lily_moe_stack_prefill")


def lily_moe_stack_decode(dims, x, layers: list, eps=1e-6, layer_inputs=None,
                          layer_logits=None, ws=None, stream=None):
    """n_layers pre-norm MoE layers on the fp32 residual x [T][d] (T <= 8),
    in place."""
    arr = (Weights * len(layers))(*[l.c for l in layers])
    rc = lib().lily_moe_stack_decode(ctypes.byref(dims), len(layers), arr, _ptr(x), eps,
                                     _ptr(layer_inputs), _ptr(layer_logits), _ptr(ws), ws.numel(),
                                     _stream(stream))
    _check(rc, "lily_moe_stack_decode")


def lily_moe_status(ws, stream=None) -> int:
    rc = lib().lily_moe_status(_ptr(ws), _stream(stream))
    if rc < 0:
        raise LilyError(rc, "lily_moe_status")
    return rc


def lily_moe_set_route_wait_ns(ns: int) -> int:
    """Give-up limit of the routing kernel's grid-barrier wait; returns the
    previous limit (nanoseconds)."""
    return int(lib().lily_moe_set_route_wait_ns(int(ns)))


def lily_moe_profile_enable(on: bool = True):
    _check(lib().lily_moe_profile_enable(1 if on else 0), "lily_moe_profile_enable")


def lily_moe_profile_read() -> dict:
    ms = (ctypes.c_double * LILY_KERNEL_KINDS)()
    n = (ctypes.c_int64 * LILY_KERNEL_KINDS)()
    _check(lib().lily_moe_profile_read(ctypes.cast(ms, ctypes.c_void_p),
                                       ctypes.cast(n, ctypes.c_void_p)), "lily_moe_profile_read")
    out = {}
    for i in range(LILY_KERNEL_KINDS):
        if n[i]:
            out[lily_moe_kernel_name(i)] = {"ms": ms[i], "launches": int(n[i])}
    return out


def lily_moe_kernel_name(kind: int) -> str:
    return lib().lily_moe_kernel_name(kind).decode()


def lily_moe_version() -> str:
    return lib().lily_moe_version().decode()
