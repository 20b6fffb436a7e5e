#!/usr/bin/env python3
"""Benchmark of the W4 MoE expert layer on GB300.

One step of a layer workload = one whole MoE layer (router logits, top-k +
gates, histogram, scan, scatter, block map, gate/up grouped GEMM with fused
dequant + SwiGLU, down grouped GEMM with fused dequant + gated combine; fp32
output) over one batch of T tokens, through the library's C ABI.  One step of
the stacked workload `stack8192` = one 8192-token prompt through 40 pre-norm
MoE layers in chunks of 2048 tokens.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the FP64 CPU oracle, timed

Prints ONE JSON line (rank 0).  With --gpus N > 1 outside a launcher it runs
itself as N ranks under torch.distributed.run.  Multi-GPU runs are token data
parallel with replicated weights and no exchange: every rank runs its own
batch (weak scaling); the time is the slowest rank's.
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

def _wl(kind, T, d, E, k, F, zipf=None, bm=128, **kw):
    return dict(kind=kind, T=T, d=d, E=E, k=k, F=F, zipf=zipf, bm=bm, **kw)


WORKLOADS = {
    # one MoE layer per step
    "prefill512": _wl("layer", 512, 2048, 256, 8, 512, bm=64),
    "prefill2048": _wl("layer", 2048, 2048, 256, 8, 512),
    "prefill2048_zipf": _wl("layer", 2048, 2048, 256, 8, 512, zipf=1.1),
    "prefill8192": _wl("layer", 8192, 2048, 256, 8, 512),  # one unchunked call
    "decode1": _wl("layer", 1, 2048, 256, 8, 512),
    "decode5": _wl("layer", 5, 2048, 256, 8, 512),
    "small": _wl("layer", 32, 512, 32, 4, 128, bm=32),
    # 40 pre-norm MoE layers, an 8192-token prompt in chunks of 2048 per step
    "stack8192": _wl("stack_prefill", 8192, 2048, 256, 8, 512, layers=40, chunk=2048),
    # one decode step (T rows) through 40 pre-norm MoE layers per step
    "decode1_stack40": _wl("stack_decode", 1, 2048, 256, 8, 512, layers=40),
    "decode5_stack40": _wl("stack_decode", 5, 2048, 256, 8, 512, layers=40),
}
DEFAULT_WORKLOAD = "prefill512"

# ncu DRAM traffic (read + write bytes per launch) of the dominant kernel, keyed
# by workload and by a hash of the kernel's source files: a changed kernel
# reports null until it is profiled again.  KERNEL_SOURCES lists the sources
# each kernel family is built from.
KERNEL_SOURCES = {
    "gemm": ["w4_grouped_gemm_gb300/csrc/gemm.cu", "w4_grouped_gemm_gb300/csrc/common.cuh"],
    "decode": ["w4_grouped_gemm_gb300/csrc/decode.cu", "w4_grouped_gemm_gb300/csrc/common.cuh",
               "w4_grouped_gemm_gb300/csrc/routing.cuh"],
}


def kernel_family(name: str) -> str:
    return "decode" if name.startswith("dec_") else "gemm"


NCU_TRAFFIC = {  # {(workload, kernel, source_hash): bytes per launch}
    # ncu dram__bytes_read.sum + dram__bytes_write.sum of the dominant kernel,
    # from the launch list of `bench.py --workload W --eager --steps 3
    # --warmup 3 --layers 1 --no-cpu-baseline --no-e2e` (mean over launches)
    ("prefill512", "gateup_gemm", "4fbc732c9698cc88"): 325353168,  # 322.25 + 3.11 MB
    ("prefill2048_zipf", "gateup_gemm", "4fbc732c9698cc88"): 227830656,  # 210.14 + 17.69 MB
    ("prefill8192", "gateup_gemm", "4fbc732c9698cc88"): 670299472,  # 605.30 + 65.00 MB
    ("decode1", "dec_router", "549388bb5c81e12a"): 3928672,  # 3.93 MB read
    ("decode1", "dec_gateup", "549388bb5c81e12a"): 10657264,  # 10.66 MB read
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


def layer_seed(layer: int, rank: int) -> int:
    """Seed of one layer's synthetic inputs on one rank: every rank draws its
    own token batch and weights (token data parallel, weak scaling)."""
    return 2000 + 3 * layer + 10000 * rank  # layer inputs draw from seed, seed+1, seed+2


def host_cpu():
    """(logical CPUs, CPU model) of this host, for the CPU-baseline record."""
    model = None
    try:
        for line in Path("/proc/cpuinfo").read_text().splitlines():
            key = line.split(":")[0].strip().lower()
            if key in ("model name", "cpu model", "hardware") and ":" in line:
                model = line.split(":", 1)[1].strip()
                break
    except OSError:
        pass
    if not model:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    return os.cpu_count(), model or "unknown"


def spawn_ranks(n: int, argv) -> int:
    """Run this script as n ranks on one node (one process per GPU) under
    torch.distributed.run, as `bench.py --gpus n` asks when no launcher set
    the rank environment; returns the launcher's exit code."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr", "127.0.0.1", f"--master-port={port}",
           str(Path(__file__).resolve())] + list(argv)
    return subprocess.call(cmd)


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
    """--impl reference: the oracle as it stands, on the host cores (rank 0
    only; under a multi-rank launch the other ranks exit without work)."""
    if rank != 0:
        return
    wl = WORKLOADS[args.workload]
    stack = wl["kind"] == "stack_prefill"
    T = wl.get("chunk", wl["T"]) if stack else wl["T"]
    shape = (T, wl["d"], wl["E"], wl["k"], wl["F"], wl["zipf"])
    nlay = wl["layers"] if stack else 1
    # one step = one token row of the workload through the oracle layer (for
    # the stacked prefill: one row of one layer, its time counted once per layer)
    n_rows = 1
    for i in range(args.warmup):
        oracle_sample(shape, 1000, n_rows, i)
    t = 0.0
    for i in range(args.steps):
        t += oracle_sample(shape, 1000, n_rows, args.warmup + i)
    t *= nlay
    value = args.steps * n_rows / t
    ncpu, model = host_cpu()
    sample = f"{n_rows} token row per step, {args.steps} steps"
    if stack:
        sample += f"; one layer's time x {nlay} layers (extrapolated)"
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload, "T": wl["T"], "d_model": wl["d"],
                   "n_experts": wl["E"], "top_k": wl["k"], "d_ff": wl["F"], "zipf_s": wl["zipf"],
                   "step_sample": f"{n_rows} token row(s) per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "nproc": ncpu, "cpu_model": model, "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


# ----------------------------------------------------------------- GPU arm
def expert_matrix_bytes(d, F):
    """One W4 matrix of one expert: packed codes + bf16 scale and bias."""
    return F * d // 2 + F * d // 64 * 4


def kernel_work(name, T, d, E, k, F, touched):
    """Algorithmic (bytes, flops) of one launch of a kernel of the layer, or
    None: weights of the touched experts (routed experts with rows + shared)
    once, activations in and out once; H, tiles and accumulators are the
    implementation's traffic and are not counted."""
    mb = expert_matrix_bytes(d, F)
    P = T * k
    if name in ("gateup_gemm", "dec_gateup"):
        return touched * 2 * mb + T * d * 2, 4 * (P + T) * d * F
    if name in ("down_gemm", "dec_down"):
        return touched * mb + T * d * 4, 2 * (P + T) * d * F
    if name in ("router_gemm", "dec_router"):
        return E * d * 4 + T * d * 2 + T * E * 4, 2 * T * d * E
    if name == "route":
        return T * E * 4 + T * k * 8, 0
    if name == "combine":  # each token's k + 1 fp16 rows in, the fp32 row out
        return (P + T) * d * 2 + T * d * 4, 0
    return None


def roofline_of(name, dur_s, work, hbm, tflops, peak_src):
    """Roofline object of one kernel: the bound whose time is longer (bytes at
    the measured copy bandwidth, or flops at the measured bf16 tensor rate --
    the fp16 kind::f16 MMAs run at the bf16 rate)."""
    nbytes, flops = work
    t_hbm = nbytes / (hbm * 1e9)
    t_tc = flops / (tflops * 1e12) if flops else 0.0
    if t_tc > t_hbm:
        achieved = flops / dur_s / 1e12
        return {"bound": "tensor", "achieved": achieved, "peak": tflops, "unit": "TFLOP/s",
                "frac": achieved / tflops, "kernel": name,
                "algorithmic_flops_per_launch": flops, "algorithmic_bytes_per_launch": nbytes,
                "peak_source": f"bf16_tflops (burst) of {peak_src} peaks"}
    achieved = nbytes / dur_s / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
            "frac": achieved / hbm, "kernel": name, "algorithmic_bytes_per_launch": nbytes,
            "algorithmic_flops_per_launch": flops,
            "peak_source": f"hbm_gbs of {peak_src} peaks (copy bandwidth)"}


def group_sizes(counts_list):
    """Rows per routed expert (the grouped GEMM's group sizes), over the
    layers a step rotates through."""
    c = np.concatenate([np.asarray(x) for x in counts_list])
    return {"min": int(c.min()), "median": float(np.median(c)), "p90": float(np.percentile(c, 90)),
            "max": int(c.max()), "empty_experts_per_layer": float((c == 0).sum() / len(counts_list)),
            "experts": int(len(counts_list[0]))}


class LayerRun:
    """One MoE layer per step (lily_moe_forward, or lily_moe_decode for T <= 8),
    rotating through several layers of weights so no step finds its weights
    in L2."""

    def __init__(self, lily, synth, wl, args, rank, dev):
        T, d, E, k, F = wl["T"], wl["d"], wl["E"], wl["k"], wl["F"]
        self.lily, self.wl, self.dev = lily, wl, dev
        self.decode = T <= 8
        shape = synth.LayerShape(T, d, E, k, F)
        self.dims = lily.make_dims(T, d, E, k, F, args.tile_rows)
        # prefill weights are 455 MB a layer; decode touches ~16 MB a layer, so
        # its timed runs rotate >= 16 layers to stay well above the 126 MB L2
        # (eager runs, used for profiling, take --layers as given)
        self.nl = max(args.layers, 16) if self.decode and not args.eager else args.layers
        self.layers = []
        for l in range(self.nl):
            inp = synth.make_layer(shape, layer_seed(l, rank), device=dev, zipf_s=wl["zipf"])
            w = lily.LayerWeights(inp["router_w"], inp["router_b"], inp["experts"])
            if T > 8:  # weights are static: their router split is made once, at load
                w.split_router()
            self.layers.append((inp["x"], w))
        self.r = lily.RoutingBuffers(self.dims, dev)
        self.ws = lily.alloc_workspace(lily.lily_moe_workspace_bytes(self.dims), dev)
        self.y = torch.empty(T, d, dtype=lily.out_torch_dtype(self.dims), device=dev)
        self.call = lily.lily_moe_decode if self.decode else lily.lily_moe_forward
        self.tokens_per_step = T
        self.rotation = self.nl
        self.counts = []

    def step(self, i):
        x, w = self.layers[i % self.nl]
        self.call(self.dims, x, w, self.r, self.y, self.ws, None)

    def after_warmup(self):
        for l in range(self.nl):
            self.step(l)
            torch.cuda.synchronize()
            self.counts.append(self.r.counts.cpu().numpy().copy())

    def status(self):
        return self.lily.lily_moe_status(self.ws)


    def touched(self):
        return float(np.mean([(c > 0).sum() + 1 for c in self.counts]))

    def layer_work(self):
        wl, T = self.wl, self.wl["T"]
        d, F, E = wl["d"], wl["F"], wl["E"]
        nbytes = self.touched() * 3 * expert_matrix_bytes(d, F) + E * d * 4 + T * d * (2 + 4)
        return nbytes, layer_flops(T, d, E, wl["k"], F), self.nl

    # end to end: host x in, the layer through the host-buffer entry point, host y
    # out, every step.  Prefill keeps two calls in flight on two streams (each
    # with its own staging, routing buffers, workspace and host output), so one
    # call's copies overlap the other's kernels; its kernels fill the GPU, so
    # the kernels of the two calls still run one after the other.  Decode runs
    # one synchronous call at a time: two T = 1 layers in flight would share
    # the GPU as a batch of two, a different workload.
    def e2e_prepare(self):
        T, d = self.wl["T"], self.wl["d"]
        self.xh = [self.layers[l][0].cpu().pin_memory() for l in range(self.nl)]
        nsets = 1 if self.decode else 2
        self.e2e_sets = []
        for j in range(nsets):
            first = j == 0
            self.e2e_sets.append({
                "r": self.r if first else self.lily.RoutingBuffers(self.dims, self.dev),
                "ws": self.ws if first else self.lily.alloc_workspace(
                    self.lily.lily_moe_workspace_bytes(self.dims), self.dev),
                "y": self.y if first else torch.empty_like(self.y),
                "xd": torch.empty(T, d, dtype=torch.bfloat16, device=self.dev),
                "yh": torch.empty(T, d, dtype=self.y.dtype).pin_memory(),
                "stream": None if self.decode else torch.cuda.Stream(device=self.dev),
                "busy": False})
        # every (layer, buffer set) pair is called once before timing (its
        # first call runs eagerly and captures the graph later calls replay)
        self.e2e_warm = max(3, self.nl * nsets)
        self.h2d = T * d * 2
        self.d2h = T * d * self.y.element_size()

    def e2e_step(self, i):
        b = self.e2e_sets[i % len(self.e2e_sets)]
        x, w = self.xh[i % self.nl], self.layers[i % self.nl][1]
        if b["stream"] is None:
            self.lily.lily_moe_forward_host(self.dims, x, b["xd"], w, b["r"], b["y"], b["yh"],
                                            b["ws"], None)
            return
        if b["busy"]:
            b["stream"].synchronize()  # this set's previous call has finished
        self.lily.lily_moe_forward_host_async(self.dims, x, b["xd"], w, b["r"], b["y"], b["yh"],
                                              b["ws"], b["stream"])
        b["busy"] = True

    def e2e_drain(self):
        for b in self.e2e_sets:
            if b["stream"] is not None and b["busy"]:
                b["stream"].synchronize()
                b["busy"] = False
        for b in self.e2e_sets:
            if self.lily.lily_moe_status(b["ws"]):
                raise RuntimeError("device status bits set in the end-to-end leg")

    def config(self):
        c = {"l2": f"inputs larger than L2: {self.nl} layers of weights rotated per step",
             "path": "decode GEMV" if self.decode else "prefill grouped GEMM",
             "experts_touched_per_step": self.touched(),
             "expert_group_rows": group_sizes(self.counts)}
        return c


class StackPrefillRun:
    """The stacked-layer prefill: one step is one T_total-token prompt through
    n_layers pre-norm MoE layers with an fp32 residual, in chunks of `chunk`
    tokens (lily_moe_stack_prefill).  The 40 layers' weights (18.2 GB) dwarf
    L2.  Each step first restores the prompt's input x (one device copy of
    T_total * d fp32, 64 MB, about 0.1% of a step), because the call updates x
    in place."""

    def __init__(self, lily, synth, wl, args, rank, dev):
        d, E, k, F = wl["d"], wl["E"], wl["k"], wl["F"]
        self.lily, self.wl, self.dev = lily, wl, dev
        self.chunk, self.T_total, self.nlay = wl["chunk"], wl["T"], wl["layers"]
        self.dims = lily.make_dims(self.chunk, d, E, k, F, args.tile_rows)
        self.weights = []
        for l in range(self.nlay):
            wr, br = synth.make_router(E, d, layer_seed(l, rank) + 1, dev)
            ex = synth.make_experts(E, d, F, layer_seed(l, rank) + 2, dev)
            self.weights.append(lily.LayerWeights(wr, br, ex).split_router())
        g = torch.Generator(device=dev)
        g.manual_seed(layer_seed(0, rank))
        self.x0 = torch.randn(self.T_total, d, generator=g, device=dev, dtype=torch.float32)
        self.x = self.x0.clone()
        self.ws = lily.alloc_workspace(lily.lily_moe_stack_workspace_bytes(self.dims), dev)
        self.tokens_per_step = self.T_total
        self.rotation = 1
        self.nchunks = self.T_total // self.chunk
        self.touched_l = []

    def step(self, i):
        self.x.copy_(self.x0)
        self.lily.lily_moe_stack_prefill(self.dims, self.x, self.weights, 1e-6, None, None,
                                         self.ws, None)

    def after_warmup(self):
        # experts touched per (layer, chunk), from one traced pass
        E, d = self.wl["E"], self.wl["d"]
        logits = torch.empty(self.nlay, self.T_total, E, dtype=torch.float32, device=self.dev)
        self.x.copy_(self.x0)
        self.lily.lily_moe_stack_prefill(self.dims, self.x, self.weights, 1e-6, None, logits,
                                         self.ws, None)
        torch.cuda.synchronize()
        k = self.wl["k"]
        top = torch.topk(logits.view(self.nlay, self.nchunks, self.chunk, E), k, dim=-1).indices
        for l in range(self.nlay):
            for c in range(self.nchunks):
                self.touched_l.append(int(torch.unique(top[l, c]).numel()) + 1)
        del logits

    def status(self):
        return self.lily.lily_moe_status(self.ws)


    def touched(self):
        return float(np.mean(self.touched_l))

    def layer_work(self):
        wl = self.wl
        d, F, E, k = wl["d"], wl["F"], wl["E"], wl["k"]
        per = self.touched() * 3 * expert_matrix_bytes(d, F) + E * d * 4 + self.chunk * d * 12
        n = self.nlay * self.nchunks
        return per * n, layer_flops(self.chunk, d, E, k, F) * n, 1

    def e2e_prepare(self):
        self.xh = self.x0.cpu().pin_memory()
        self.xo = torch.empty_like(self.xh).pin_memory()
        self.h2d = self.xh.numel() * 4
        self.d2h = self.xo.numel() * 4

    def e2e_step(self, i):
        self.x.copy_(self.xh, non_blocking=True)
        self.lily.lily_moe_stack_prefill(self.dims, self.x, self.weights, 1e-6, None, None,
                                         self.ws, None)
        self.xo.copy_(self.x, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    def config(self):
        return {"l2": f"inputs larger than L2: {self.nlay} layers of weights (18.2 GB) per step",
                "path": "stacked prefill (pre-norm MoE layers, fp32 residual)",
                "layers": self.nlay, "chunk_tokens": self.chunk, "prompt_tokens": self.T_total,
                "experts_touched_per_layer_chunk": self.touched(),
                "step_restores_input": "one 64 MB device copy of x per step"}


class StackDecodeRun:
    """The stacked decode step: one step is T rows (one token of T sequences,
    or a speculative-verify batch) through n_layers pre-norm MoE layers with
    an fp32 residual, every launch chained on the device
    (lily_moe_stack_decode).  The step reads each layer's router and touched
    experts (~18 MB a layer at T=1; 40 layers: far above L2).  Each step first
    restores the input x (a T * d fp32 device copy), because the call updates
    x in place."""

    def __init__(self, lily, synth, wl, args, rank, dev):
        T, d, E, k, F = wl["T"], wl["d"], wl["E"], wl["k"], wl["F"]
        self.lily, self.wl, self.dev = lily, wl, dev
        self.nlay = wl["layers"]
        self.dims = lily.make_dims(T, d, E, k, F, args.tile_rows)
        self.weights = []
        for l in range(self.nlay):
            wr, br = synth.make_router(E, d, layer_seed(l, rank) + 1, dev)
            ex = synth.make_experts(E, d, F, layer_seed(l, rank) + 2, dev)
            self.weights.append(lily.LayerWeights(wr, br, ex))
        g = torch.Generator(device=dev)
        g.manual_seed(layer_seed(0, rank))
        self.x0 = torch.randn(T, d, generator=g, device=dev, dtype=torch.float32)
        self.x = self.x0.clone()
        self.ws = lily.alloc_workspace(lily.lily_moe_stack_workspace_bytes(self.dims), dev)
        self.tokens_per_step = T
        self.rotation = 1
        self.touched_l = []

    def step(self, i):
        self.x.copy_(self.x0)
        self.lily.lily_moe_stack_decode(self.dims, self.x, self.weights, 1e-6, None, None,
                                        self.ws, None)

    def after_warmup(self):
        T, E, k = self.wl["T"], self.wl["E"], self.wl["k"]
        logits = torch.empty(self.nlay, T, E, dtype=torch.float32, device=self.dev)
        self.x.copy_(self.x0)
        self.lily.lily_moe_stack_decode(self.dims, self.x, self.weights, 1e-6, None, logits,
                                        self.ws, None)
        torch.cuda.synchronize()
        top = torch.topk(logits, k, dim=-1).indices
        for l in range(self.nlay):
            self.touched_l.append(int(torch.unique(top[l]).numel()) + 1)

    def status(self):
        return self.lily.lily_moe_status(self.ws)

    def touched(self):
        return float(np.mean(self.touched_l))

    def layer_work(self):
        wl = self.wl
        T, d, F, E, k = wl["T"], wl["d"], wl["F"], wl["E"], wl["k"]
        per = self.touched() * 3 * expert_matrix_bytes(d, F) + E * d * 4 + T * d * 8
        return per * self.nlay, layer_flops(T, d, E, k, F) * self.nlay, 1

    def e2e_prepare(self):
        self.xh = self.x0.cpu().pin_memory()
        self.xo = torch.empty_like(self.xh).pin_memory()
        self.h2d = self.xh.numel() * 4
        self.d2h = self.xo.numel() * 4

    def e2e_step(self, i):
        self.x.copy_(self.xh, non_blocking=True)
        self.lily.lily_moe_stack_decode(self.dims, self.x, self.weights, 1e-6, None, None,
                                        self.ws, None)
        self.xo.copy_(self.x, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    def config(self):
        return {"l2": f"inputs larger than L2: {self.nlay} layers' routers and touched experts "
                      f"per step", "path": "stacked decode (pre-norm MoE layers, fp32 residual)",
                "layers": self.nlay, "experts_touched_per_layer": self.touched(),
                "step_us": None, "step_restores_input": "one T x d fp32 device copy per step"}


def run_lily(args, world, rank, local):
    import w4_grouped_gemm_gb300 as lily
    from w4_grouped_gemm_gb300 import synth

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lily.lib()
    wl = WORKLOADS[args.workload]
    T, d, E, k, F = wl["T"], wl["d"], wl["E"], wl["k"], wl["F"]
    run = {"layer": LayerRun, "stack_prefill": StackPrefillRun,
           "stack_decode": StackDecodeRun}[wl["kind"]](
        lily, synth, wl, args, rank, dev)
    stream = torch.cuda.current_stream(dev)

    for i in range(args.warmup):
        run.step(i)
    torch.cuda.synchronize()
    if run.status() != 0:
        raise RuntimeError("device status bits set during warm-up")
    run.after_warmup()

    # The timed steps replay CUDA graphs of the C-ABI calls: one graph of
    # `rotation` consecutive steps replayed steps // rotation times, then one
    # of the remaining steps, so exactly `steps` steps run; eager launches if
    # capture is not possible.
    rot = run.rotation
    reps, rem = divmod(args.steps, rot)
    graphs = None
    if not args.eager:
        try:
            graphs = []
            for n in (rot if reps else 0, rem):
                if n == 0:
                    graphs.append(None)
                    continue
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    for i in range(n):
                        run.step(i)
                g.replay()
                graphs.append(g)
            torch.cuda.synchronize()
        except Exception as exc:  # noqa: BLE001
            print(f"graph capture unavailable ({exc}); timing eager launches", file=sys.stderr)
            graphs = None
            torch.cuda.synchronize()

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
    if graphs is not None:
        for _ in range(reps):
            graphs[0].replay()
        if graphs[1] is not None:
            graphs[1].replay()
    else:
        for i in range(args.steps):
            run.step(i)
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
    del graphs

    # Per-kernel device time: the library's CUDA events around every kernel,
    # recorded on the launch stream, in a captured graph of the same steps
    # replayed once (eager when no graph).
    prof_steps = max(1, min(args.steps, 10 * rot))
    lily.lily_moe_profile_enable(True)
    lily.lily_moe_profile_read()
    for i in range(prof_steps):  # eager pass: also fills the library's event pool
        run.step(i)
    torch.cuda.synchronize()
    prof = lily.lily_moe_profile_read()
    if not args.eager:
        try:
            pgraph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(pgraph):
                for i in range(prof_steps):
                    run.step(i)
            pgraph.replay()  # its event records now hold this replay's times
            torch.cuda.synchronize()
            prof = lily.lily_moe_profile_read()
            del pgraph
        except Exception as exc:  # noqa: BLE001
            print(f"profiled graph unavailable ({exc}); eager per-kernel times", file=sys.stderr)
    lily.lily_moe_profile_enable(False)
    status = run.status()
    if status:
        raise RuntimeError(f"device status bits set: {status}")

    # end to end through the public API with host buffers
    run.e2e_prepare()
    e2e_steps = 3 if args.no_e2e else max(3, min(args.steps, 5 if wl["kind"] == "stack_prefill"
                                                  else 200))
    for i in range(getattr(run, "e2e_warm", 3)):
        run.e2e_step(i)
    if hasattr(run, "e2e_drain"):
        run.e2e_drain()
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        run.e2e_step(i)
    if hasattr(run, "e2e_drain"):
        run.e2e_drain()  # the last calls' results are in host memory
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(e2e_s, world, dev)

    if rank != 0:
        return
    hbm, tf_burst, tf_sus, peak_src = measured_peaks()
    tps = run.tokens_per_step
    value = job_throughput(world, tps, args.steps, ms / 1000.0)
    e2e_value = job_throughput(world, tps, e2e_steps, e2e_s)
    step_s = ms / 1000.0 / args.steps
    step_bytes, step_flops, _ = run.layer_work()
    step_t_hbm = step_bytes / (hbm * 1e9)
    step_t_tc = step_flops / (tf_sus * 1e12)
    total_ms = sum(u["ms"] for u in prof.values())
    kernels = {n: {"us_per_launch": 1e3 * v["ms"] / v["launches"], "launches": v["launches"],
                   "share": v["ms"] / total_ms} for n, v in prof.items()}
    dom = max(prof, key=lambda n: prof[n]["ms"]) if prof else None
    roofline = None
    touched = run.touched()
    chunk_T = run.dims.T
    for n in kernels:
        work = kernel_work(n, chunk_T, d, E, k, F, touched)
        if work:
            rf = roofline_of(n, kernels[n]["us_per_launch"] * 1e-6, work, hbm, tf_burst, peak_src)
            kernels[n]["bound"], kernels[n]["frac"] = rf["bound"], rf["frac"]
    if dom:
        work = kernel_work(dom, chunk_T, d, E, k, F, touched)
        if work:
            roofline = roofline_of(dom, kernels[dom]["us_per_launch"] * 1e-6, work, hbm, tf_burst,
                                   peak_src)
            roofline["traffic"] = NCU_TRAFFIC.get(
                (args.workload, dom, source_hash(KERNEL_SOURCES[kernel_family(dom)])))
    launches = int(round(sum(v["launches"] for v in prof.values()) / prof_steps * args.steps))
    clocks = sampler.summary(t_wall0, t_wall1) if sampler else None

    # CPU baseline: the oracle, bounded sample of the same workload
    cpu = None
    if not args.no_cpu_baseline:
        ncpu, model = host_cpu()
        layer_shape = (chunk_T, d, E, k, F, wl["zipf"])
        if wl["kind"] == "stack_prefill":
            n_rows = args.cpu_rows
            t_cpu = oracle_sample(layer_shape, 1000, n_rows)
            nl = wl["layers"]
            cpu = {"value": n_rows / (t_cpu * nl), "unit": UNIT, "cores": 1, "kind": "oracle",
                   "nproc": ncpu, "cpu_model": model, "extrapolated": True,
                   "sample": f"{n_rows} token rows of one {chunk_T}-token layer, time x {nl} "
                             f"layers (extrapolated: the prompt is {nl} layers x "
                             f"{run.nchunks} chunks of {chunk_T} tokens)"}
        else:
            n_rows = 1 if run.decode else args.cpu_rows
            t_cpu = oracle_sample(layer_shape, 1000, n_rows)
            cpu = {"value": n_rows / t_cpu, "unit": UNIT, "cores": 1, "kind": "oracle",
                   "nproc": ncpu, "cpu_model": model,
                   "sample": f"{n_rows} token rows of the {args.workload} layer (router logits, "
                             f"routing, explicit dequant of every touched expert, FP64 layer)"}
    cfg = {"workload": args.workload, "T": T, "d_model": d, "n_experts": E, "top_k": k,
           "d_ff": F, "zipf_s": wl["zipf"], "tile_rows": args.tile_rows,
           "launch": "CUDA graph replay of the C-ABI calls" if not args.eager else "eager",
           "parallelism": f"token data parallel x{world} (replicated weights, no exchange)",
           "step_algorithmic_bytes": step_bytes, "step_flops": step_flops,
           "step_roofline_us": 1e6 * max(step_t_hbm, step_t_tc),
           "step_frac_of_roofline": max(step_t_hbm, step_t_tc) / step_s,
           "step_bound": "tensor" if step_t_tc > step_t_hbm else "hbm",
           "kernels": kernels}
    cfg.update(run.config())
    if "step_us" in cfg:
        cfg["step_us"] = 1e3 * ms / args.steps
        cfg["layer_us"] = cfg["step_us"] / wl["layers"]
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "f16 tensor-core operands (W4 weights, bf16 x), fp32 accumulate, fp32 out",
        "data": "synthetic (seeded; shapes and distributions of the workload)",
        "config": cfg,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": run.h2d,
                "d2h_bytes_per_step": run.d2h},
        "gpu_launches": launches,
        "clocks": clocks,
    }
    print(json.dumps(out), flush=True)


class Ablation:
    """The two bench-only ablations of design points of the path, on one
    seeded prefill layer (shape `shape`, tile rows BM):
      host_routing -- routing on the GPU, then a host sync, a copy of the
        counts to the host, the block map built on the host and copied back,
        then the expert GEMMs (lily_moe_experts);
      dequant_hbm -- every expert's weights dequantised to fp16 in HBM each
        step (torch element-wise ops: unpack, then one multiply-add pass),
        then batched fp16 GEMMs (torch.bmm, cuBLAS) over expert-padded rows,
        with the same GPU routing.
    fused() runs the library's layer into y_ref, run(name) an ablation into
    y; both fp32 [T][d]."""

    def __init__(self, lily, synth, shape, BM, seed, dev, zipf=None):
        T, d, E, k, F = shape.T, shape.d, shape.E, shape.k, shape.F
        self.lily, self.shape, self.BM, self.dev = lily, shape, BM, dev
        self.dims = lily.make_dims(T, d, E, k, F, BM)
        self.inp = synth.make_layer(shape, seed, device=dev, zipf_s=zipf)
        self.x = self.inp["x"]
        self.w = lily.LayerWeights(self.inp["router_w"], self.inp["router_b"], self.inp["experts"])
        if T > 8:
            self.w.split_router()
        self.r = lily.RoutingBuffers(self.dims, dev)
        self.ws = lily.alloc_workspace(lily.lily_moe_workspace_bytes(self.dims), dev)
        self.y_ref = torch.empty(T, d, dtype=torch.float32, device=dev)
        self.y = torch.empty_like(self.y_ref)
        self.cap = lily.lily_moe_block_map_cap(self.dims)

    def fused(self):
        self.lily.lily_moe_forward(self.dims, self.x, self.w, self.r, self.y_ref, self.ws)

    def run(self, name):
        getattr(self, name)()

    def host_routing(self):
        lily, r, E, BM = self.lily, self.r, self.shape.E, self.BM
        lily.lily_moe_route(self.dims, self.x, None, self.w, r, self.ws)
        counts = r.counts.cpu().numpy()  # waits for the routing, copies to the host
        off = np.concatenate([[0], np.cumsum(counts)])
        tiles = [(e, off[e] + i * BM) for e in range(E) for i in range(-(-int(counts[e]) // BM))]
        bm = np.full((self.cap, 2), -1, np.int32)
        bm[:len(tiles)] = np.asarray(tiles, np.int32).reshape(-1, 2)
        r.block_map.copy_(torch.from_numpy(bm))
        r.n_tiles.fill_(len(tiles))
        lily.lily_moe_experts(self.dims, self.x, self.w, r, self.y, self.ws)

    @staticmethod
    def _deq(q, sc, bi):  # fp16 [n][rows][cols] = scale * q + bias, in HBM
        n, rows, half = q.shape
        qq = torch.stack((q & 15, q >> 4), dim=-1).view(n, rows, half * 2 // 64, 64).half()
        return torch.addcmul(bi.half()[..., None], qq, sc.half()[..., None]).view(n, rows, -1)

    def dequant_hbm(self):
        lily, r, dev = self.lily, self.r, self.dev
        T, d, E, k = self.shape.T, self.shape.d, self.shape.E, self.shape.k
        P, ex, y, x = T * k, self.inp["experts"], self.y, self.x
        lily.lily_moe_route(self.dims, x, None, self.w, r, self.ws)
        wg = self._deq(ex["gate_q"], ex["gate_s"], ex["gate_b"])
        wu = self._deq(ex["up_q"], ex["up_s"], ex["up_b"])
        wd = self._deq(ex["down_q"], ex["down_s"], ex["down_b"])
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


def run_ablation(args, world, rank, local):
    """Bench-only ablations (Ablation), each timed eagerly against the fused
    path in the same run (one JSON line), with its output checked against the
    fused path's."""
    import w4_grouped_gemm_gb300 as lily
    from w4_grouped_gemm_gb300 import synth

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = WORKLOADS[args.workload]
    T, d, E, k, F, zipf = wl["T"], wl["d"], wl["E"], wl["k"], wl["F"], wl["zipf"]
    if T <= 8 or wl["kind"] != "layer":
        raise SystemExit("ablations are single-layer prefill only")
    ab = Ablation(lily, synth, synth.LayerShape(T, d, E, k, F), args.tile_rows, layer_seed(0, 0),
                  dev, zipf)
    y, y_ref, ex, BM = ab.y, ab.y_ref, ab.inp["experts"], args.tile_rows
    fused = ab.fused

    def timed(fn, n):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n):
            fn()
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / n

    abl = getattr(ab, args.ablation)
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
    ap.add_argument("--tile-rows", type=int, default=None,
                    help="block-map tile rows BM (default: the workload's, 64 at T=512, else 128)")
    ap.add_argument("--layers", type=int, default=4)
    ap.add_argument("--cpu-rows", type=int, default=64)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg (profiling)")
    ap.add_argument("--eager", action="store_true", help="time eager launches, no CUDA graph")
    ap.add_argument("--ablation", choices=["host_routing", "dequant_hbm"], default=None,
                    help="bench-only ablation of a design point (prefill workloads)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.tile_rows is None:
        args.tile_rows = WORKLOADS[args.workload]["bm"]
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(spawn_ranks(args.gpus, sys.argv[1:]))
    world, rank, local = dist_info()
    if args.gpus != world:
        raise SystemExit(f"--gpus {args.gpus} but {world} rank(s) were launched")
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
