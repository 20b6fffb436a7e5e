#!/usr/bin/env python3
"""Benchmark of the W4 MoE expert layer on GB300.

One step = one whole MoE layer (router logits, top-k + gates, histogram,
scan, scatter, block map, gate/up grouped GEMM with fused dequant + SwiGLU,
down grouped GEMM with fused dequant + gated combine, bf16 output) over one
batch of T tokens, through the library's C ABI.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the FP64 CPU oracle, timed

Prints ONE JSON line (rank 0).  Multi-GPU runs (torchrun) are token data
parallel with replicated weights and no exchange: every rank runs its own
batch (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "MoE-layer tokens/s"
UNIT = "tokens/s"

WORKLOADS = {
    # name: (T, d, E, k, F, zipf)
    "prefill512": (512, 2048, 256, 8, 512, None),
    "prefill2048_zipf": (2048, 2048, 256, 8, 512, 1.1),
    "prefill2048": (2048, 2048, 256, 8, 512, None),
    "decode1": (1, 2048, 256, 8, 512, None),
    "decode5": (5, 2048, 256, 8, 512, None),
    "prefill8192": (8192, 2048, 256, 8, 512, None),  # one unchunked call
    "small": (32, 512, 32, 4, 128, None),
}
DEFAULT_WORKLOAD = "prefill512"

# ncu DRAM traffic (read + write bytes per launch) of the dominant kernel, keyed
# by workload and by a hash of the kernel's source files: a changed kernel
# reports null until it is profiled again.
KERNEL_SOURCES = ["w4_grouped_gemm_gb300/csrc/gemm.cu", "w4_grouped_gemm_gb300/csrc/common.cuh"]
NCU_TRAFFIC = {  # {(workload, kernel, source_hash): bytes}
    # ncu dram__bytes_{read,write}.sum, w4_gemm_kernel<1, 64>, prefill512 layer:
    # 322.20 MB read + 6.06 MB written
    ("prefill512", "gateup_gemm", "fe4c349ddb1b7603"): 328253440,
}


def source_hash(files) -> str:
    h = hashlib.sha256()
    for f in files:
        h.update((ROOT / f).read_bytes())
    return h.hexdigest()[:16]


def measured_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return d.get("hbm_gbs"), d.get("bf16_tflops"), d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 50):
        self.index = index
        self.period_ms = period_ms
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (FileNotFoundError, OSError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)

    def summary(self, t0=None, t1=None):
        rows = []
        for ts, line in self.lines:
            if t0 is not None and not (t0 - 0.25 <= ts <= t1 + 0.25):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------- helpers
def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest value over all ranks (the job's time is its slowest rank's)."""
    if world <= 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, tokens_per_rank: int, steps: int, seconds: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank * steps / seconds


def algorithmic_bytes(T, d, E, k, F, counts, y_bytes=4):
    """Touched experts' W4 bytes (packed + bf16 scale/bias) + router W + x + y."""
    per_expert = 3 * (F * d // 2 + F * d // 64 * 4)
    touched = int((np.asarray(counts) > 0).sum()) + 1  # + shared expert
    return touched * per_expert + E * d * 4 + T * d * (2 + y_bytes), touched


def gateup_bytes(T, d, F, touched):
    """Gate/up kernel: touched experts' gate+up W4 bytes + x read."""
    return touched * 2 * (F * d // 2 + F * d // 64 * 4) + T * d * 2


def layer_flops(T, d, E, k, F):
    return 2 * T * d * E + T * (k + 1) * 6 * d * F


# ----------------------------------------------------------------- CPU oracle
def oracle_sample(shape_args, seed, n_rows, rows_offset=0):
    """Time the FP64 oracle on a bounded sample of the workload: router logits,
    routing and the layer output of n_rows tokens (host inputs)."""
    import oracle
    from w4_grouped_gemm_gb300 import synth
    T, d, E, k, F, zipf = shape_args
    shape = synth.LayerShape(T, d, E, k, F)
    inp = synth.make_layer(shape, seed, device="cpu", zipf_s=zipf)
    x = synth.bf16_bits(inp["x"])
    wr = inp["router_w"].numpy()
    br = None if inp["router_b"] is None else inp["router_b"].numpy()
    w = synth.experts_to_numpy(inp["experts"])
    rows = (np.arange(n_rows) + rows_offset) % T
    oracle.build()
    t0 = time.perf_counter()
    L, _ = oracle.router_logits(x[rows], wr, br)
    ro = oracle.route(L.astype(np.float32), k, 128)
    oracle.moe_rows(x[rows], w, ro["ids"], ro["gates"], np.arange(n_rows))
    return time.perf_counter() - t0


def run_reference(args, ws, rank):
    """--impl reference: the oracle as it stands, on the host cores."""
    if rank != 0:
        return
    wl = WORKLOADS[args.workload]
    T, d, E, k, F, zipf = wl
    # one step = one token row of the workload through the oracle layer
    n_rows = 1
    for i in range(args.warmup):
        oracle_sample(wl, 1000, n_rows, i)
    t = 0.0
    for i in range(args.steps):
        t += oracle_sample(wl, 1000, n_rows, args.warmup + i)
    value = args.steps * n_rows / t
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload, "T": T, "d_model": d, "n_experts": E, "top_k": k,
                   "d_ff": F, "zipf_s": zipf, "step_sample": f"{n_rows} token row(s) per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{n_rows} token row per step, {args.steps} steps"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


# ----------------------------------------------------------------- GPU arm
def run_lily(args, world, rank, local):
    import w4_grouped_gemm_gb300 as lily
    from w4_grouped_gemm_gb300 import synth

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lily.lib()
    T, d, E, k, F, zipf = WORKLOADS[args.workload]
    decode = T <= 8
    shape = synth.LayerShape(T, d, E, k, F)
    dims = lily.make_dims(T, d, E, k, F, args.tile_rows)
    # several layers of weights, rotated per step, so no step finds the
    # previous step's weights in L2 (each layer's weights are 455 MB)
    # decode touches ~16 MB per layer: rotate >= 16 layers so no step finds
    # its weights in the 126 MB L2
    nl = max(args.layers, 16) if decode else args.layers
    layers = []
    for l in range(nl):
        inp = synth.make_layer(shape, 1000 * 2 + 17 * l + 101 * rank, device=dev, zipf_s=zipf)
        layers.append((inp["x"], lily.LayerWeights(inp["router_w"], inp["router_b"], inp["experts"])))
    r = lily.RoutingBuffers(dims, dev)
    wsb = lily.alloc_workspace(lily.lily_moe_workspace_bytes(dims), dev)
    y = torch.empty(T, d, dtype=lily.out_torch_dtype(dims), device=dev)
    stream = torch.cuda.current_stream(dev)
    call = lily.lily_moe_decode if decode else lily.lily_moe_forward

    def step(i):  # on the current stream (the capture stream inside a graph)
        x, w = layers[i % nl]
        call(dims, x, w, r, y, wsb, None)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if lily.lily_moe_status(wsb) != 0:
        raise RuntimeError("device status bits set during warm-up")
    counts_by_layer = []
    for l in range(nl):
        step(l)
        torch.cuda.synchronize()
        counts_by_layer.append(r.counts.cpu().numpy().copy())

    # The timed steps replay a CUDA graph of the C-ABI calls (one command
    # buffer per group of nl layer steps), so host submission does not gate
    # the device; fall back to eager launches if capture is not possible.
    graph = None
    if not args.eager:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for i in range(nl):
                    step(i)
            graph.replay()
            torch.cuda.synchronize()
        except Exception as exc:  # noqa: BLE001
            print(f"graph capture unavailable ({exc}); timing eager launches", file=sys.stderr)
            graph = None
            torch.cuda.synchronize()
    reps = max(1, args.steps // nl) if graph is not None else args.steps
    steps_timed = reps * nl if graph is not None else args.steps

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t_wall0 = time.perf_counter()
    e0.record(stream)
    if graph is not None:
        for _ in range(reps):
            graph.replay()
    else:
        for i in range(args.steps):
            step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.perf_counter()
    if world > 1:
        torch.distributed.barrier()
    ms = e0.elapsed_time(e1)
    if sampler:
        time.sleep(0.2)
        sampler.stop()
    ms = max_over_ranks(ms, world, dev)
    args.steps = steps_timed

    # Per-kernel device time: the library's CUDA events around every kernel,
    # recorded on the launch stream.  The same steps are captured with the
    # event records inside the graph and replayed once (eager when no graph).
    prof_steps = min(steps_timed, 40 * nl)
    lily.lily_moe_profile_enable(True)
    lily.lily_moe_profile_read()
    for i in range(prof_steps):  # eager pass: also fills the library's event pool
        step(i)
    torch.cuda.synchronize()
    prof = lily.lily_moe_profile_read()
    if graph is not None:
        try:
            pgraph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(pgraph):
                for i in range(prof_steps):
                    step(i)
            pgraph.replay()  # its event records now hold this replay's times
            torch.cuda.synchronize()
            prof = lily.lily_moe_profile_read()
            del pgraph
        except Exception as exc:  # noqa: BLE001
            print(f"profiled graph unavailable ({exc}); eager per-kernel times", file=sys.stderr)
    lily.lily_moe_profile_enable(False)
    status = lily.lily_moe_status(wsb)
    if status:
        raise RuntimeError(f"device status bits set: {status}")

    # end to end through the host-buffer entry point (pinned host x and y)
    e2e_steps = 3 if args.no_e2e else max(3, min(args.steps, 200))
    xh = [layers[l][0].cpu().pin_memory() for l in range(nl)]
    yh = torch.empty(T, d, dtype=y.dtype).pin_memory()
    xd = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    for i in range(3):
        lily.lily_moe_forward_host(dims, xh[i % nl], xd, layers[i % nl][1], r, y, yh, wsb, stream)
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        lily.lily_moe_forward_host(dims, xh[i % nl], xd, layers[i % nl][1], r, y, yh, wsb, stream)
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(e2e_s, world, dev)

    if rank != 0:
        return
    hbm, tf_burst, tf_sus, peak_src = measured_peaks()
    value = job_throughput(world, T, args.steps, ms / 1000.0)
    e2e_value = job_throughput(world, T, e2e_steps, e2e_s)
    alg_bytes = []
    touched_l = []
    for c in counts_by_layer:
        b, tch = algorithmic_bytes(T, d, E, k, F, c)
        alg_bytes.append(b)
        touched_l.append(tch)
    step_bytes = float(np.mean(alg_bytes))
    flops = layer_flops(T, d, E, k, F)
    step_s = ms / 1000.0 / args.steps
    layer_t_hbm = step_bytes / (hbm * 1e9)
    layer_t_tc = flops / (tf_sus * 1e12)
    # dominant kernel of the step by device time
    kernels = {n: {"ms_per_launch": v["ms"] / v["launches"], "launches": v["launches"],
                   "share": v["ms"] / sum(u["ms"] for u in prof.values())}
               for n, v in prof.items()}
    dom = max(prof, key=lambda n: prof[n]["ms"]) if prof else None
    roofline = None
    if dom:
        dur = prof[dom]["ms"] / prof[dom]["launches"] / 1000.0
        touched = float(np.mean(touched_l))
        if dom == "gateup_gemm":
            dbytes = gateup_bytes(T, d, F, touched)
        elif dom == "down_gemm":
            dbytes = touched * (F * d // 2 + F * d // 64 * 4) + T * d * 2
        elif dom in ("dec_gateup",):
            dbytes = gateup_bytes(T, d, F, touched)
        elif dom in ("dec_down_combine",):
            dbytes = touched * (F * d // 2 + F * d // 64 * 4)
        elif dom in ("router_gemv", "router_gemm"):
            dbytes = E * d * 4 + T * d * 2  # router weights (fp32) and x
        else:
            dbytes = step_bytes
        achieved = dbytes / dur / 1e9
        key = (args.workload, dom, source_hash(KERNEL_SOURCES))
        roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                    "frac": achieved / hbm, "traffic": NCU_TRAFFIC.get(key),
                    "kernel": dom, "algorithmic_bytes_per_launch": dbytes,
                    "peak_source": f"hbm_gbs of {peak_src} peaks (copy bandwidth)"}
    per_step = sum(v["launches"] for n, v in prof.items() if n != "memset_acc") / max(prof_steps, 1)
    launches = int(round(per_step * args.steps))
    clocks = sampler.summary(t_wall0, t_wall1) if sampler else None

    # CPU baseline: the oracle, bounded sample of the same workload
    cpu = None
    if not args.no_cpu_baseline:
        n_rows = 1 if decode else args.cpu_rows
        t_cpu = oracle_sample(WORKLOADS[args.workload], 1000, n_rows)
        cpu = {"value": n_rows / t_cpu, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{n_rows} token rows of the {args.workload} layer (router logits, "
                         f"routing, explicit dequant of every touched expert, FP64 layer)"}
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16 tensor-core operands (W4 weights, bf16 x), fp32 accumulate, fp32 out",
        "data": "synthetic (seeded; shapes and distributions of the workload)",
        "config": {
            "workload": args.workload, "T": T, "d_model": d, "n_experts": E, "top_k": k,
            "d_ff": F, "zipf_s": zipf, "tile_rows": args.tile_rows,
            "path": "decode GEMV" if decode else "prefill grouped GEMM",
            "l2": f"inputs larger than L2: {nl} layers of weights rotated per step",
            "launch": "CUDA graph replay of the C-ABI calls" if graph is not None else "eager",
            "parallelism": f"token data parallel x{world} (replicated weights, no exchange)",
            "experts_touched_per_step": float(np.mean(touched_l)),
            "layer_algorithmic_bytes": step_bytes, "layer_flops": flops,
            "layer_roofline_us": 1e6 * max(layer_t_hbm, layer_t_tc),
            "layer_frac_of_roofline": max(layer_t_hbm, layer_t_tc) / step_s,
            "kernels": kernels,
        },
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": T * d * 2,
                "d2h_bytes_per_step": T * d * y.element_size()},
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if decode and graph is not None:
        # the graph replays nl consecutive layers (each its own weights, chained
        # with programmatic dependent launch): one token through an nl-layer
        # MoE stack
        out["config"]["stack_layers"] = nl
        out["config"]["stack_step_us"] = 1e3 * ms / args.steps * nl
    print(json.dumps(out), flush=True)


def run_ablation(args, world, rank, local):
    """Bench-only ablations of two design points of the path, each timed eagerly
    against the fused path in the same run (one JSON line):
      host_routing -- routing on the GPU, then a host sync, a copy of the
        counts to the host, the block map built on the host and copied back,
        then the expert GEMMs (lily_moe_experts);
      dequant_hbm -- every expert's weights dequantised to fp16 in HBM each
        step (torch element-wise ops: unpack, then one multiply-add pass),
        then batched fp16 GEMMs (torch.bmm, cuBLAS) over expert-padded rows,
        with the same GPU routing.
    Both check their layer output against the fused path's."""
    import w4_grouped_gemm_gb300 as lily
    from w4_grouped_gemm_gb300 import synth

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    T, d, E, k, F, zipf = WORKLOADS[args.workload]
    if T <= 8:
        raise SystemExit("ablations are prefill-only")
    shape = synth.LayerShape(T, d, E, k, F)
    dims = lily.make_dims(T, d, E, k, F, args.tile_rows)
    inp = synth.make_layer(shape, 1000 * 2 + 17, device=dev, zipf_s=zipf)
    x = inp["x"]
    w = lily.LayerWeights(inp["router_w"], inp["router_b"], inp["experts"])
    r = lily.RoutingBuffers(dims, dev)
    ws = lily.alloc_workspace(lily.lily_moe_workspace_bytes(dims), dev)
    y_ref = torch.empty(T, d, dtype=torch.float32, device=dev)
    y = torch.empty_like(y_ref)
    BM, P, cap = args.tile_rows, T * k, lily.lily_moe_block_map_cap(dims)

    def fused():
        lily.lily_moe_forward(dims, x, w, r, y_ref, ws)

    def host_routing():
        lily.lily_moe_route(dims, x, None, w, r, ws)
        counts = r.counts.cpu().numpy()  # waits for the routing, copies to the host
        off = np.concatenate([[0], np.cumsum(counts)])
        tiles = [(e, off[e] + i * BM) for e in range(E) for i in range(-(-int(counts[e]) // BM))]
        bm = np.full((cap, 2), -1, np.int32)
        bm[:len(tiles)] = np.asarray(tiles, np.int32).reshape(-1, 2)
        r.block_map.copy_(torch.from_numpy(bm))
        r.n_tiles.fill_(len(tiles))
        lily.lily_moe_experts(dims, x, w, r, y, ws)

    ex = inp["experts"]

    def deq(q, sc, bi):  # fp16 [n][rows][cols] = scale * q + bias, in HBM
        n, rows, half = q.shape
        qq = torch.stack((q & 15, q >> 4), dim=-1).view(n, rows, half * 2 // 64, 64).half()
        return torch.addcmul(bi.half()[..., None], qq, sc.half()[..., None]).view(n, rows, -1)

    def dequant_hbm():
        lily.lily_moe_route(dims, x, None, w, r, ws)
        wg = deq(ex["gate_q"], ex["gate_s"], ex["gate_b"])
        wu = deq(ex["up_q"], ex["up_s"], ex["up_b"])
        wd = deq(ex["down_q"], ex["down_s"], ex["down_b"])
        pad = int(r.counts.max())
        pos = torch.arange(P, device=dev)
        e_of = torch.searchsorted(r.offsets[1:].contiguous(), pos.int(), right=True)
        slot = pos - r.offsets[e_of].long()
        p = r.perm.long()
        tok = p // k
        gate = r.topk_gates.reshape(-1)[p]
        xh = x.half()
        X = torch.zeros(E, pad, d, dtype=torch.half, device=dev)
        X[e_of, slot] = xh[tok]
        H = torch.nn.functional.silu(torch.bmm(X, wg[:E].transpose(1, 2))) * torch.bmm(
            X, wu[:E].transpose(1, 2))
        O = torch.bmm(H, wd[:E].transpose(1, 2))
        y.zero_()
        y.index_add_(0, tok, O[e_of, slot].float() * gate[:, None])
        hs = torch.nn.functional.silu(xh @ wg[E].t()) * (xh @ wu[E].t())
        y.add_((hs @ wd[E].t()).float())

    def timed(fn, n):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n):
            fn()
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / n

    abl = {"host_routing": host_routing, "dequant_hbm": dequant_hbm}[args.ablation]
    n = max(3, min(args.steps, 50))
    t_fused = timed(fused, n)
    t_abl = timed(abl, n)
    fused()
    abl()
    torch.cuda.synchronize()
    err = float((y - y_ref).abs().max() / y_ref.pow(2).mean().sqrt())
    floor_us = None
    if args.ablation == "dequant_hbm":
        # HBM floor of this path whatever its kernels: read the packed weights,
        # write them as fp16, read the fp16 weights back in the GEMMs
        hbm, _, _, _ = measured_peaks()
        packed = sum(t.numel() * t.element_size() for t in ex.values())
        fp16 = sum(t.numel() * 2 * 2 for n, t in ex.items() if n.endswith("_q"))
        floor_us = 1e6 * (packed + 2 * fp16) / (hbm * 1e9)
    out = {
        "metric": METRIC, "value": T / t_abl, "unit": UNIT, "n_gpus": 1, "steps": n,
        "warmup": 3, "ms_per_step": 1e3 * t_abl, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp16 weights in HBM" if args.ablation == "dequant_hbm"
        else "f16 tensor-core operands (W4 weights, bf16 x), fp32 accumulate, fp32 out",
        "data": "synthetic (seeded; shapes and distributions of the workload)",
        "impl": "lily", "ablation": args.ablation,
        "config": {"workload": args.workload, "T": T, "tile_rows": BM, "launch": "eager",
                   "fused_eager_us": 1e6 * t_fused, "ablation_us": 1e6 * t_abl,
                   "slowdown_vs_fused": t_abl / t_fused,
                   "max_err_vs_fused_over_rms": err, "hbm_floor_us": floor_us},
    }
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["lily", "reference"], default="lily")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--tile-rows", type=int, default=64)
    ap.add_argument("--layers", type=int, default=4)
    ap.add_argument("--cpu-rows", type=int, default=64)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg (profiling)")
    ap.add_argument("--eager", action="store_true", help="time eager launches, no CUDA graph")
    ap.add_argument("--ablation", choices=["host_routing", "dequant_hbm"], default=None,
                    help="bench-only ablation of a design point (prefill workloads)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_info()
    if world > 1:
        backend = "nccl" if torch.cuda.is_available() and args.impl == "lily" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        torch.distributed.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        elif args.ablation:
            run_ablation(args, world, rank, local)
        else:
            run_lily(args, world, rank, local)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
