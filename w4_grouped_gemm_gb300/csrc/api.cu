// api.cu -- the C ABI (include/lily_moe.h): argument validation, workspace
// layout and the launch sequence of each call.  No call allocates device
// memory; every launch goes to the caller's stream.
#include <array>
#include <atomic>
#include <cstring>
#include <map>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace lily {

// ---------------------------------------------------------------- profiling
namespace {
struct ProfRec {
  int kind;
  cudaEvent_t a, b;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof_open;  // recorded, not yet read
std::vector<cudaEvent_t> g_prof_pool;
int g_prof_kind = -1;
cudaEvent_t g_prof_start = nullptr;

// Record e on s; inside a stream capture the record must be an external
// event-record node so that it records each time the graph runs.
void prof_record(cudaEvent_t e, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
  else
    cudaEventRecord(e, s);
}

cudaEvent_t prof_event() {
  if (!g_prof_pool.empty()) {
    cudaEvent_t e = g_prof_pool.back();
    g_prof_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}
}  // namespace

void prof_begin(int kind, cudaStream_t s) {
  if (!g_prof_on) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_kind = kind;
  g_prof_start = prof_event();
  prof_record(g_prof_start, s);
}

void prof_end(int kind, cudaStream_t s) {
  if (!g_prof_on) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (g_prof_kind != kind || !g_prof_start) return;
  cudaEvent_t e = prof_event();
  prof_record(e, s);
  g_prof_open.push_back({kind, g_prof_start, e});
  g_prof_start = nullptr;
  g_prof_kind = -1;
}

// ---------------------------------------------------------------- wait limit
namespace {
std::atomic<uint64_t> g_route_wait_ns{2000000000ull};
}
uint64_t route_wait_limit_ns() { return g_route_wait_ns.load(std::memory_order_relaxed); }

// ---------------------------------------------------------------- host caches
namespace {
std::mutex g_attr_mu;
std::map<std::pair<int, const void*>, size_t> g_smem_set;
}  // namespace

cudaError_t ensure_smem_attr(const void* func, size_t bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_attr_mu);
  auto key = std::make_pair(dev, func);
  auto it = g_smem_set.find(key);
  if (it != g_smem_set.end() && it->second >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) g_smem_set[key] = bytes;
  return e;
}

// ---------------------------------------------------------------- workspace
namespace {

constexpr size_t kAlign = 256;
inline size_t up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

struct Layout {
  size_t ctrl, hist, x16, xs, w3, part, H, O, tiles, plan, total;
};

// ctrl: [0] status, [1] grid-barrier count, [2] grid-barrier generation,
// [3] decode router CTAs done
Layout layout(const lily_moe_dims& d) {
  const size_t T = d.T, E = d.n_experts, k = d.top_k, F = d.d_ff, D = d.d_model;
  const size_t P = T * k;
  const size_t nblk = (size_t)route_blocks((int)T);
  Layout L;
  size_t off = 0;
  L.ctrl = off; off += up(256);
  L.hist = off; off += up(nblk * E * 4);
  L.x16 = off;  off += up(T * D * 2);
  L.xs = off;   off += up(P * D * 2);
  const bool tc_router = d.T > 8;  // tensor-core router: split W + split-K partials
  L.w3 = off;   off += tc_router ? up(3 * E * D * 2) : 0;
  L.part = off; off += tc_router ? up((size_t)router_splits(d.T, d.d_model) * T * E * 4) : 0;
  L.H = off;    off += up((P + T) * F * 2);
  L.O = off;    off += up((P + T) * D * 2);  // grouped GEMM path: the down GEMM's rows
  L.tiles = off; off += up((size_t)tile_count(d.T, d.n_experts, d.top_k, d.tile_rows) * 16);
  L.plan = off;  off += d.T <= 8 ? up(decode_plan_bytes()) : 0;  // decode: the step's slots
  L.total = off;
  return L;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Compute capability 10.3 of the current device, checked once per device.
int check_arch() {
  static int arch_seen[64] = {};  // 0 unknown, 1 sm_103, -1 other
  int dev = 0, maj = 0, min = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LILY_ERR_CUDA;
  if (dev >= 0 && dev < 64 && arch_seen[dev]) return arch_seen[dev] > 0 ? LILY_OK : LILY_ERR_ARCH;
  if (cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return LILY_ERR_CUDA;
  const bool ok = maj == 10 && min == 3;
  if (dev >= 0 && dev < 64) arch_seen[dev] = ok ? 1 : -1;
  return ok ? LILY_OK : LILY_ERR_ARCH;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? LILY_OK : LILY_ERR_CUDA; }

int check_routing(const lily_moe_routing* r) {
  if (!r) return LILY_ERR_INVALID_ARG;
  const void* ptrs[] = {r->logits, r->topk_ids, r->topk_gates, r->counts, r->offsets,
                        r->perm,   r->inv_perm, r->block_map,  r->n_tiles};
  for (const void* p : ptrs) {
    if (!p) return LILY_ERR_INVALID_ARG;
    if (!aligned16(p)) return LILY_ERR_MISALIGNED;
  }
  return LILY_OK;
}

int check_weights(const lily_moe_weights* w, bool need_router, bool need_experts) {
  if (!w) return LILY_ERR_INVALID_ARG;
  if (need_router) {
    if (!w->router_w) return LILY_ERR_INVALID_ARG;
    if (!aligned16(w->router_w) || (w->router_bias && !aligned16(w->router_bias)) ||
        (w->router_w_split && !aligned16(w->router_w_split)))
      return LILY_ERR_MISALIGNED;
  }
  if (need_experts) {
    const void* ptrs[] = {w->gate_q, w->gate_s, w->gate_b, w->up_q,  w->up_s,
                          w->up_b,   w->down_q, w->down_s, w->down_b};
    for (const void* p : ptrs) {
      if (!p) return LILY_ERR_INVALID_ARG;
      if (!aligned16(p)) return LILY_ERR_MISALIGNED;
    }
  }
  return LILY_OK;
}

int check_ws(const lily_moe_dims* d, void* ws, size_t bytes) {
  if (!ws) return LILY_ERR_INVALID_ARG;
  if (!aligned16(ws)) return LILY_ERR_MISALIGNED;
  if (bytes < layout(*d).total) return LILY_ERR_WORKSPACE_TOO_SMALL;
  return LILY_OK;
}

uint32_t* ws_status(void* ws) { return reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws)); }

RouteArgs route_args(const lily_moe_dims& d, const float* logits_in, const lily_moe_routing& r,
                     void* ws) {
  const Layout L = layout(d);
  uint8_t* base = static_cast<uint8_t*>(ws);
  uint32_t* ctrl = reinterpret_cast<uint32_t*>(base + L.ctrl);
  RouteArgs a;
  a.logits_src = logits_in ? logits_in : r.logits;
  a.logits_dst = r.logits;
  a.T = d.T;
  a.E = d.n_experts;
  a.k = d.top_k;
  a.BM = d.tile_rows;
  a.cap = (int)lily_moe_block_map_cap(&d);
  a.ids = r.topk_ids;
  a.gates = r.topk_gates;
  a.counts = r.counts;
  a.offsets = r.offsets;
  a.perm = r.perm;
  a.inv = r.inv_perm;
  a.block_map = r.block_map;
  a.n_tiles = r.n_tiles;
  a.hist = reinterpret_cast<int32_t*>(base + L.hist);
  a.bar = ctrl + 1;
  a.status = ws_status(ws);
  a.wait_ns = route_wait_limit_ns();
  return a;
}

// The decode router (T <= 8): logits, x in the decode GEMV's fragment order
// in the x16 / xs regions, and (its last CTA) the routing outputs and the
// step's plan.  With norm (the stacked decode) x is the fp32 residual and the
// router scores bf16(rmsnorm(x, eps)).
int do_dec_router(const lily_moe_dims& d, const void* x, const lily_moe_weights* w,
                  const lily_moe_routing& r, void* ws, cudaStream_t s, bool norm = false,
                  float eps = 0.f) {
  const Layout L = layout(d);
  uint8_t* base = static_cast<uint8_t*>(ws);
  DecRouterArgs da = {};
  da.x = x;
  da.w = w->router_w;
  da.b = w->router_bias;
  da.logits = r.logits;
  da.xpg = reinterpret_cast<uint32_t*>(base + L.x16);
  da.xsg = reinterpret_cast<float*>(base + L.xs);
  da.eps = eps;
  da.T = d.T;
  da.d = d.d_model;
  da.E = d.n_experts;
  da.route = route_args(d, nullptr, r, ws);
  da.plan = base + L.plan;
  da.done = reinterpret_cast<uint32_t*>(base + L.ctrl) + 3;
  // (routing-only calls may pass no expert weights: then nothing is prefetched)
  const bool experts = w->gate_q && w->gate_s && w->gate_b && w->up_q && w->up_s && w->up_b &&
                       w->down_q && w->down_s && w->down_b;
  da.F = experts ? d.d_ff : 0;
  da.gq = w->gate_q; da.gs = w->gate_s; da.gb = w->gate_b;
  da.uq = w->up_q;   da.us = w->up_s;   da.ub = w->up_b;
  da.dq = w->down_q; da.ds = w->down_s; da.db = w->down_b;
  return cuda_rc(launch_dec_router(da, norm, s));
}

// Routing on `s`: router logits (unless logits_in is given), then the
// routing kernel.  No host synchronisation.
int do_route(const lily_moe_dims& d, const void* x, const float* logits_in,
             const lily_moe_weights* w, const lily_moe_routing& r, void* ws, cudaStream_t s) {
  const Layout L = layout(d);
  uint8_t* base = static_cast<uint8_t*>(ws);
  if (!logits_in) {
    if (d.T > 8) {
      float* part = reinterpret_cast<float*>(base + L.part);
      cudaError_t e = launch_router_tc(x, w->router_w, w->router_bias, d.T, d.d_model,
                                       d.n_experts, base + L.w3, w->router_w_split, part,
                                       r.logits, ws_status(ws), s);
      if (e != cudaSuccess) return LILY_ERR_CUDA;
    } else {
      return do_dec_router(d, x, w, r, ws, s);  // routes in its last CTA
    }
  }
  return cuda_rc(launch_route(route_args(d, logits_in, r, ws), s));
}

GemmArgs gemm_args(const lily_moe_dims& d, const lily_moe_weights* w, const lily_moe_routing& r,
                   void* ws) {
  const Layout L = layout(d);
  uint8_t* base = static_cast<uint8_t*>(ws);
  GemmArgs a;
  a.T = d.T;
  a.E = d.n_experts;
  a.k = d.top_k;
  a.d = d.d_model;
  a.F = d.d_ff;
  a.BM = d.tile_rows;
  a.block_map = r.block_map;
  a.n_tiles = r.n_tiles;
  a.offsets = r.offsets;
  a.perm = r.perm;
  a.gates = r.topk_gates;
  a.s0 = w->gate_s;
  a.b0 = w->gate_b;
  a.s1 = w->up_s;
  a.b1 = w->up_b;
  a.inv = r.inv_perm;
  a.H = base + L.H;
  a.O = base + L.O;
  a.tiles = reinterpret_cast<int4*>(base + L.tiles);
  a.status = ws_status(ws);
  return a;
}

// The grouped GEMMs (token rows, gate/up + SwiGLU, down) from routing
// already in r, then the combine of each token's rows: into y (fp32 or bf16
// per d.out_dtype), or -- with resid -- added to the fp32 residual with the
// next layer's RMSNorm into xn (when xn is non-NULL).
int do_experts(const lily_moe_dims& d, const void* x, const lily_moe_weights* w,
               const lily_moe_routing& r, void* ws, cudaStream_t s, void* y,
               float* resid = nullptr, void* xn = nullptr, float eps = 0.f) {
  GemmArgs a = gemm_args(d, w, r, ws);
  const Layout L = layout(d);
  uint8_t* base = static_cast<uint8_t*>(ws);
  if (launch_token_rows(a, x, base + L.xs, base + L.x16, s) != cudaSuccess) return LILY_ERR_CUDA;
  if (launch_gateup(a, base + L.xs, base + L.x16, w->gate_q, w->up_q, s) != cudaSuccess)
    return LILY_ERR_CUDA;
  a.s0 = w->down_s;
  a.b0 = w->down_b;
  a.s1 = nullptr;
  a.b1 = nullptr;
  if (launch_down(a, w->down_q, s) != cudaSuccess) return LILY_ERR_CUDA;
  return cuda_rc(launch_combine(a, y, d.out_dtype == LILY_DTYPE_F32, resid, xn, eps, s));
}

// Arguments of the decode GEMV launches (after do_route for T <= 8): the
// layer output goes to y, or is added to the fp32 residual `resid`.
DecodeArgs decode_args(const lily_moe_dims& d, const lily_moe_weights* w,
                       const lily_moe_routing& r, void* ws, void* y, float* resid) {
  const Layout L = layout(d);
  uint8_t* base = static_cast<uint8_t*>(ws);
  DecodeArgs a;
  a.T = d.T;
  a.E = d.n_experts;
  a.k = d.top_k;
  a.d = d.d_model;
  a.F = d.d_ff;
  a.BM = d.tile_rows;
  a.cap = (int)lily_moe_block_map_cap(&d);
  a.plan = base + L.plan;
  a.gq = w->gate_q; a.gs = w->gate_s; a.gb = w->gate_b;
  a.uq = w->up_q;   a.us = w->up_s;   a.ub = w->up_b;
  a.dq = w->down_q; a.ds = w->down_s; a.db = w->down_b;
  a.xpg = reinterpret_cast<const uint32_t*>(base + L.x16);
  a.xsg = reinterpret_cast<const float*>(base + L.xs);
  a.H = base + L.H;
  a.y = y;
  a.y_f32 = d.out_dtype == LILY_DTYPE_F32;
  a.resid = resid;
  a.status = ws_status(ws);
  return a;
}

// Routing + grouped GEMMs + combine.
int do_forward(const lily_moe_dims& d, const void* x, const lily_moe_weights* w,
               const lily_moe_routing& r, void* ws, cudaStream_t s, void* y,
               float* resid = nullptr, void* xn = nullptr, float eps = 0.f) {
  const int rc = do_route(d, x, nullptr, w, r, ws, s);
  if (rc) return rc;
  return do_experts(d, x, w, r, ws, s, y, resid, xn, eps);
}

int common_checks(const lily_moe_dims* dims, const void* x, const lily_moe_weights* w,
                  const lily_moe_routing* r, const void* y, void* ws, size_t ws_bytes,
                  bool experts) {
  if (!dims) return LILY_ERR_INVALID_ARG;
  int rc = lily_moe_check_dims(dims);
  if (rc) return rc;
  if (!x || (experts && !y)) return LILY_ERR_INVALID_ARG;
  if (!aligned16(x) || (y && !aligned16(y))) return LILY_ERR_MISALIGNED;
  if ((rc = check_weights(w, true, experts))) return rc;
  if ((rc = check_routing(r))) return rc;
  if ((rc = check_ws(dims, ws, ws_bytes))) return rc;
  return check_arch();
}

// ---- end-to-end calls: host buffers in and out

size_t host_x_bytes(const lily_moe_dims& d) { return (size_t)d.T * d.d_model * 2; }
size_t host_y_bytes(const lily_moe_dims& d) {
  return (size_t)d.T * d.d_model * (d.out_dtype == LILY_DTYPE_F32 ? 4 : 2);
}

// Whether a host buffer is page-locked (cudaHostAlloc / cudaHostRegister):
// only such copies can be captured in a graph.  (Copies by the SMs through the
// buffer's device mapping were measured slower than the copy engines at every
// size from 4 KB to 8 MB, so the copy engines move the data either way.)
bool host_pinned(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeHost;
}

struct HostStep {
  const lily_moe_dims* dims;
  const void* x_host;
  void* x_dev;
  const lily_moe_weights* w;
  lily_moe_routing* r;
  void* y_dev;
  void* y_host;
  void* ws;
  size_t ws_bytes;
};

// Copy in, run the layer, copy out, all on `s` (no synchronisation).
int host_step(const HostStep& h, cudaStream_t s) {
  if (cudaMemcpyAsync(h.x_dev, h.x_host, host_x_bytes(*h.dims), cudaMemcpyHostToDevice, s) !=
      cudaSuccess)
    return LILY_ERR_CUDA;
  const int rc = h.dims->T <= 8
                     ? lily_moe_decode(h.dims, h.x_dev, h.w, h.r, h.y_dev, h.ws, h.ws_bytes, s)
                     : lily_moe_forward(h.dims, h.x_dev, h.w, h.r, h.y_dev, h.ws, h.ws_bytes, s);
  if (rc) return rc;
  return cuda_rc(
      cudaMemcpyAsync(h.y_host, h.y_dev, host_y_bytes(*h.dims), cudaMemcpyDeviceToHost, s));
}

// Instantiated graphs of host_step, one per argument set (dims, every pointer,
// the device), least recently used evicted.  A graph reads its buffers by
// address, so their contents may change freely between calls.  The capacity
// holds one graph per layer of a deep stack called layer by layer.
using HostGraphKey = std::array<uint64_t, 40>;
struct HostGraph {
  cudaGraphExec_t exec;  // nullptr: capture failed, these arguments run eagerly
  uint64_t used;
};
constexpr size_t kHostGraphs = 128;
std::mutex g_hg_mu;
bool g_hg_on = true;
uint64_t g_hg_tick = 0;
std::map<HostGraphKey, HostGraph> g_hg;
std::map<int, cudaStream_t> g_hg_streams;  // capture stream per device

HostGraphKey host_graph_key(const HostStep& h) {
  HostGraphKey k{};
  size_t n = 0;
  auto put = [&](uint64_t v) { k[n++] = v; };
  auto ptr = [&](const void* p) { put((uint64_t)(uintptr_t)p); };
  const lily_moe_dims& d = *h.dims;
  for (int32_t v : {d.T, d.d_model, d.n_experts, d.top_k, d.d_ff, d.group, d.tile_rows,
                    d.out_dtype})
    put((uint64_t)(uint32_t)v);
  for (const void* p : {h.x_host, (const void*)h.x_dev, (const void*)h.y_dev,
                        (const void*)h.y_host, (const void*)h.ws})
    ptr(p);
  put((uint64_t)h.ws_bytes);
  const lily_moe_weights& w = *h.w;
  for (const void* p : {(const void*)w.router_w, (const void*)w.router_bias,
                        (const void*)w.gate_q, (const void*)w.gate_s, (const void*)w.gate_b,
                        (const void*)w.up_q, (const void*)w.up_s, (const void*)w.up_b,
                        (const void*)w.down_q, (const void*)w.down_s, (const void*)w.down_b})
    ptr(p);
  const lily_moe_routing& r = *h.r;
  for (const void* p : {(const void*)r.logits, (const void*)r.topk_ids,
                        (const void*)r.topk_gates, (const void*)r.counts, (const void*)r.offsets,
                        (const void*)r.perm, (const void*)r.inv_perm, (const void*)r.block_map,
                        (const void*)r.n_tiles})
    ptr(p);
  int dev = -1;
  cudaGetDevice(&dev);
  put((uint64_t)(uint32_t)dev);
  return k;  // 8 + 5 + 1 + 11 + 9 + 1 = 35 words used
}

// Capture host_step for these arguments on the library's own stream (the
// caller's may be the legacy default stream, which cannot be captured) and
// keep the instantiated graph; a failed capture is remembered as such.
void host_graph_capture(const HostStep& h, const HostGraphKey& key) {
  std::lock_guard<std::mutex> lk(g_hg_mu);
  if (!g_hg_on || g_hg.count(key)) return;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return;
  }
  cudaStream_t& cs = g_hg_streams[dev];
  if (!cs && cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) {
    cs = nullptr;
    cudaGetLastError();
    return;
  }
  cudaGraphExec_t exec = nullptr;
  cudaGraph_t g = nullptr;
  if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) == cudaSuccess) {
    const int rc = host_step(h, cs);
    const cudaError_t e = cudaStreamEndCapture(cs, &g);
    if (rc == LILY_OK && e == cudaSuccess && g &&
        cudaGraphInstantiate(&exec, g, 0) != cudaSuccess)
      exec = nullptr;
    if (g) cudaGraphDestroy(g);
  }
  cudaGetLastError();  // a refused capture leaves no error for the next call
  if (g_hg.size() >= kHostGraphs) {
    auto lru = g_hg.begin();
    for (auto it = g_hg.begin(); it != g_hg.end(); ++it)
      if (it->second.used < lru->second.used) lru = it;
    if (lru->second.exec) cudaGraphExecDestroy(lru->second.exec);
    g_hg.erase(lru);
  }
  g_hg[key] = {exec, ++g_hg_tick};
}

}  // namespace
}  // namespace lily

using namespace lily;

extern "C" {

int lily_moe_check_dims(const lily_moe_dims* d) {
  if (!d) return LILY_ERR_INVALID_ARG;
  if (d->T < 1 || d->d_model < 1 || d->n_experts < 1 || d->top_k < 1 || d->d_ff < 1)
    return LILY_ERR_INVALID_ARG;
  if (d->T > 16384) return LILY_ERR_UNSUPPORTED_SHAPE;
  if (d->d_model % 128 || d->d_model > 4096) return LILY_ERR_UNSUPPORTED_SHAPE;
  if (d->d_ff % 128 || d->d_ff > 4096) return LILY_ERR_UNSUPPORTED_SHAPE;
  if (d->n_experts > 256) return LILY_ERR_UNSUPPORTED_SHAPE;
  if (d->top_k > 8 || d->top_k > d->n_experts) return LILY_ERR_UNSUPPORTED_SHAPE;
  if (d->group != 64) return LILY_ERR_UNSUPPORTED_SHAPE;
  if (d->out_dtype != LILY_DTYPE_BF16 && d->out_dtype != LILY_DTYPE_F32)
    return LILY_ERR_UNSUPPORTED_SHAPE;
  if (d->tile_rows != 16 && d->tile_rows != 32 && d->tile_rows != 64 && d->tile_rows != 128)
    return LILY_ERR_UNSUPPORTED_SHAPE;
  if (gemm_stages(true, d->tile_rows, d->d_model, d->d_ff) < 2 ||
      gemm_stages(false, d->tile_rows, d->d_ff, d->d_model) < 2)
    return LILY_ERR_UNSUPPORTED_SHAPE;
  return LILY_OK;
}

size_t lily_moe_workspace_bytes(const lily_moe_dims* d) {
  if (lily_moe_check_dims(d) != LILY_OK) return 0;
  return layout(*d).total;
}

int64_t lily_moe_block_map_cap(const lily_moe_dims* d) {
  if (!d || d->tile_rows < 1 || d->T < 0 || d->top_k < 1) return 0;
  const int64_t P = (int64_t)d->T * d->top_k;
  return (P + d->tile_rows - 1) / d->tile_rows + (d->n_experts < P ? d->n_experts : P);
}

int lily_moe_route(const lily_moe_dims* dims, const void* x, const float* logits_in,
                   const lily_moe_weights* w, lily_moe_routing* r, void* ws, size_t ws_bytes,
                   void* stream) {
  if (!dims) return LILY_ERR_INVALID_ARG;
  int rc = lily_moe_check_dims(dims);
  if (rc) return rc;
  if (logits_in) {
    if (!aligned16(logits_in)) return LILY_ERR_MISALIGNED;
  } else {
    if (!x) return LILY_ERR_INVALID_ARG;
    if (!aligned16(x)) return LILY_ERR_MISALIGNED;
    if ((rc = check_weights(w, true, false))) return rc;
  }
  if ((rc = check_routing(r))) return rc;
  if ((rc = check_ws(dims, ws, ws_bytes))) return rc;
  if ((rc = check_arch())) return rc;
  const int maxb = route_max_blocks();
  if (maxb > 0 && route_blocks(dims->T) > maxb) return LILY_ERR_UNSUPPORTED_SHAPE;
  return do_route(*dims, x, logits_in, w, *r, ws, (cudaStream_t)stream);
}

int lily_moe_experts(const lily_moe_dims* dims, const void* x, const lily_moe_weights* w,
                     const lily_moe_routing* r, void* y, void* ws, size_t ws_bytes, void* stream) {
  int rc = common_checks(dims, x, w, r, y, ws, ws_bytes, true);
  if (rc) return rc;
  return do_experts(*dims, x, w, *r, ws, (cudaStream_t)stream, y);
}

int lily_moe_forward(const lily_moe_dims* dims, const void* x, const lily_moe_weights* w,
                     lily_moe_routing* r, void* y, void* ws, size_t ws_bytes, void* stream) {
  int rc = common_checks(dims, x, w, r, y, ws, ws_bytes, true);
  if (rc) return rc;
  const int maxb = route_max_blocks();
  if (maxb > 0 && route_blocks(dims->T) > maxb) return LILY_ERR_UNSUPPORTED_SHAPE;
  return do_forward(*dims, x, w, *r, ws, (cudaStream_t)stream, y);
}

int lily_moe_decode(const lily_moe_dims* dims, const void* x, const lily_moe_weights* w,
                    lily_moe_routing* r, void* y, void* ws, size_t ws_bytes, void* stream) {
  int rc = common_checks(dims, x, w, r, y, ws, ws_bytes, true);
  if (rc) return rc;
  if (dims->T > 8) return LILY_ERR_UNSUPPORTED_SHAPE;
  cudaStream_t s = (cudaStream_t)stream;
  // router logits, then the GEMVs, which route from them (three launches)
  if ((rc = do_dec_router(*dims, x, w, *r, ws, s))) return rc;
  return cuda_rc(launch_decode(decode_args(*dims, w, *r, ws, y, nullptr), s));
}

// The host-buffer step; `sync`: wait for it before returning (a replayed
// graph is otherwise left running on the stream).
static int forward_host(const lily_moe_dims* dims, const void* x_host, void* x_dev,
                        const lily_moe_weights* w, lily_moe_routing* r, void* y_dev, void* y_host,
                        void* ws, size_t ws_bytes, void* stream, bool sync) {
  if (!dims || !x_host || !y_host) return LILY_ERR_INVALID_ARG;
  int rc = common_checks(dims, x_dev, w, r, y_dev, ws, ws_bytes, true);
  if (rc) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  const HostStep h = {dims, x_host, x_dev, w, r, y_dev, y_host, ws, ws_bytes};
  bool prof;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    prof = g_prof_on;
  }
  // Pinned buffers on both sides: replay this argument set's graph, or run
  // the step eagerly and then capture one for the next call.
  const bool graphable = !prof && host_pinned(x_host) && host_pinned(y_host);
  HostGraphKey key{};
  if (graphable) {
    key = host_graph_key(h);
    int launched = 0;  // 1 launched, -1 launch failed
    {
      // launched under the lock: an eviction may destroy the graph only
      // after its launch is queued (destruction then waits for it)
      std::lock_guard<std::mutex> lk(g_hg_mu);
      auto it = g_hg_on ? g_hg.find(key) : g_hg.end();
      if (it != g_hg.end() && it->second.exec) {  // (none: capture failed, run eagerly)
        it->second.used = ++g_hg_tick;
        launched = cudaGraphLaunch(it->second.exec, s) == cudaSuccess ? 1 : -1;
      }
    }
    if (launched < 0) return LILY_ERR_CUDA;
    if (launched > 0) return sync ? cuda_rc(cudaStreamSynchronize(s)) : LILY_OK;
  }
  if ((rc = host_step(h, s))) return rc;
  if ((rc = cuda_rc(cudaStreamSynchronize(s)))) return rc;
  if (graphable) host_graph_capture(h, key);
  return LILY_OK;
}

int lily_moe_forward_host(const lily_moe_dims* dims, const void* x_host, void* x_dev,
                          const lily_moe_weights* w, lily_moe_routing* r, void* y_dev,
                          void* y_host, void* ws, size_t ws_bytes, void* stream) {
  return forward_host(dims, x_host, x_dev, w, r, y_dev, y_host, ws, ws_bytes, stream, true);
}

int lily_moe_forward_host_async(const lily_moe_dims* dims, const void* x_host, void* x_dev,
                                const lily_moe_weights* w, lily_moe_routing* r, void* y_dev,
                                void* y_host, void* ws, size_t ws_bytes, void* stream) {
  return forward_host(dims, x_host, x_dev, w, r, y_dev, y_host, ws, ws_bytes, stream, false);
}

int lily_moe_host_graphs(int enable) {
  std::lock_guard<std::mutex> lk(g_hg_mu);
  const int was = g_hg_on ? 1 : 0;
  for (auto& e : g_hg)
    if (e.second.exec) cudaGraphExecDestroy(e.second.exec);
  g_hg.clear();
  g_hg_on = enable != 0;
  return was;
}

size_t lily_moe_router_split_bytes(int32_t n_experts, int32_t d_model) {
  if (n_experts < 1 || d_model < 1) return 0;
  return (size_t)3 * n_experts * d_model * 2;
}

int lily_moe_router_split(const float* router_w, int32_t n_experts, int32_t d_model, void* split,
                          void* stream) {
  if (!router_w || !split || n_experts < 1 || n_experts > 256) return LILY_ERR_INVALID_ARG;
  if (d_model % 128 || d_model < 128 || d_model > 4096) return LILY_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(router_w) || !aligned16(split)) return LILY_ERR_MISALIGNED;
  int rc = check_arch();
  if (rc) return rc;
  return cuda_rc(launch_router_split(router_w, n_experts, d_model, split, (cudaStream_t)stream));
}

int lily_moe_rmsnorm(int32_t T, int32_t d, const float* x, float eps, void* out, void* stream) {
  if (T < 1 || d < 1 || !x || !out) return LILY_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(out)) return LILY_ERR_MISALIGNED;
  int rc = check_arch();
  if (rc) return rc;
  return cuda_rc(launch_rmsnorm(x, out, T, d, eps, (cudaStream_t)stream));
}

// Stack workspace: [layer workspace][routing buffers][xn bf16]
namespace {
struct StackLayout {
  size_t ws, logits, ids, gates, counts, offsets, perm, inv, bmap, ntiles, xn, total;
};
StackLayout stack_layout(const lily_moe_dims& d) {
  StackLayout S;
  const size_t T = d.T, E = d.n_experts, k = d.top_k, P = T * k;
  const size_t cap = (size_t)lily_moe_block_map_cap(&d);
  size_t off = 0;
  S.ws = off; off += up(layout(d).total);
  S.logits = off; off += up(T * E * 4);
  S.ids = off; off += up(P * 4);
  S.gates = off; off += up(P * 4);
  S.counts = off; off += up(E * 4);
  S.offsets = off; off += up((E + 1) * 4);
  S.perm = off; off += up(P * 4);
  S.inv = off; off += up(P * 4);
  S.bmap = off; off += up(cap * 8);
  S.ntiles = off; off += up(4);
  S.xn = off; off += up(T * d.d_model * 2);
  S.total = off;
  return S;
}
// The routing buffers of a stack workspace.
lily_moe_routing stack_routing(uint8_t* base, const StackLayout& S) {
  lily_moe_routing r;
  r.logits = reinterpret_cast<float*>(base + S.logits);
  r.topk_ids = reinterpret_cast<int32_t*>(base + S.ids);
  r.topk_gates = reinterpret_cast<float*>(base + S.gates);
  r.counts = reinterpret_cast<int32_t*>(base + S.counts);
  r.offsets = reinterpret_cast<int32_t*>(base + S.offsets);
  r.perm = reinterpret_cast<int32_t*>(base + S.perm);
  r.inv_perm = reinterpret_cast<int32_t*>(base + S.inv);
  r.block_map = reinterpret_cast<int32_t*>(base + S.bmap);
  r.n_tiles = reinterpret_cast<int32_t*>(base + S.ntiles);
  return r;
}
}  // namespace

size_t lily_moe_stack_workspace_bytes(const lily_moe_dims* d) {
  if (lily_moe_check_dims(d) != LILY_OK) return 0;
  return stack_layout(*d).total;
}

int lily_moe_stack_prefill(const lily_moe_dims* dims, int32_t T_total, int32_t n_layers,
                           const lily_moe_weights* layers, float* x, float eps,
                           float* layer_inputs, float* layer_logits, void* ws, size_t ws_bytes,
                           void* stream) {
  if (!dims || !layers || !x || !ws || n_layers < 1 || T_total < 1) return LILY_ERR_INVALID_ARG;
  int rc = lily_moe_check_dims(dims);
  if (rc) return rc;
  if (T_total % dims->T) return LILY_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || !aligned16(ws) || (layer_inputs && !aligned16(layer_inputs)) ||
      (layer_logits && !aligned16(layer_logits)))
    return LILY_ERR_MISALIGNED;
  for (int l = 0; l < n_layers; ++l)
    if ((rc = check_weights(&layers[l], true, true))) return rc;
  const StackLayout S = stack_layout(*dims);
  if (ws_bytes < S.total) return LILY_ERR_WORKSPACE_TOO_SMALL;
  if ((rc = check_arch())) return rc;
  const int T = dims->T, D = dims->d_model, E = dims->n_experts;
  if (layer_logits && ((size_t)T * E) % 4) return LILY_ERR_MISALIGNED;  // per-chunk slices
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* base = static_cast<uint8_t*>(ws);
  void* lws = base + S.ws;
  lily_moe_routing r = stack_routing(base, S);
  void* xn = base + S.xn;
  const int nchunks = T_total / T;
  for (int c = 0; c < nchunks; ++c) {
    float* xc = x + (size_t)c * T * D;
    if (launch_rmsnorm(xc, xn, T, D, eps, s) != cudaSuccess) return LILY_ERR_CUDA;
    for (int l = 0; l < n_layers; ++l) {
      if (layer_inputs &&
          cudaMemcpyAsync(layer_inputs + ((size_t)l * T_total + (size_t)c * T) * D, xc,
                          (size_t)T * D * 4, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return LILY_ERR_CUDA;
      lily_moe_routing rl = r;
      if (layer_logits) rl.logits = layer_logits + ((size_t)l * T_total + (size_t)c * T) * E;
      // the layer on bf16(rmsnorm(x)); its combine adds the output to x and
      // writes the next layer's normalised input
      if ((rc = do_forward(*dims, xn, &layers[l], rl, lws, s, nullptr, xc,
                           l + 1 < n_layers ? xn : nullptr, eps)))
        return rc;
    }
  }
  return LILY_OK;
}

int lily_moe_stack_decode(const lily_moe_dims* dims, int32_t n_layers,
                          const lily_moe_weights* layers, float* x, float eps,
                          float* layer_inputs, float* layer_logits, void* ws, size_t ws_bytes,
                          void* stream) {
  if (!dims || !layers || !x || !ws || n_layers < 1) return LILY_ERR_INVALID_ARG;
  int rc = lily_moe_check_dims(dims);
  if (rc) return rc;
  if (dims->T > 8) return LILY_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || !aligned16(ws) || (layer_inputs && !aligned16(layer_inputs)) ||
      (layer_logits && !aligned16(layer_logits)))
    return LILY_ERR_MISALIGNED;
  const int T = dims->T, D = dims->d_model, E = dims->n_experts;
  if (layer_logits && ((size_t)T * E) % 4) return LILY_ERR_MISALIGNED;  // per-layer slices
  for (int l = 0; l < n_layers; ++l)
    if ((rc = check_weights(&layers[l], true, true))) return rc;
  const StackLayout S = stack_layout(*dims);
  if (ws_bytes < S.total) return LILY_ERR_WORKSPACE_TOO_SMALL;
  if ((rc = check_arch())) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* base = static_cast<uint8_t*>(ws);
  void* lws = base + S.ws;
  lily_moe_routing r = stack_routing(base, S);
  for (int l = 0; l < n_layers; ++l) {
    if (layer_inputs &&
        cudaMemcpyAsync(layer_inputs + (size_t)l * T * D, x, (size_t)T * D * 4,
                        cudaMemcpyDeviceToDevice, s) != cudaSuccess)
      return LILY_ERR_CUDA;
    lily_moe_routing rl = r;
    if (layer_logits) rl.logits = layer_logits + (size_t)l * T * E;
    // router (on bf16(rmsnorm(x))) with the routing, then the expert GEMVs,
    // whose output is added to x: three launches per layer, each chained to
    // the previous one with programmatic dependent launch
    if ((rc = do_dec_router(*dims, x, &layers[l], rl, lws, s, true, eps))) return rc;
    if ((rc = cuda_rc(launch_decode(decode_args(*dims, &layers[l], rl, lws, nullptr, x), s))))
      return rc;
  }
  return LILY_OK;
}

int lily_moe_status(void* ws, void* stream) {
  if (!ws) return LILY_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, ws_status(ws), 4, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return LILY_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return LILY_ERR_CUDA;
  // clear the bits; after a give-up also the grid-barrier and router-done
  // counters (words 1..3), so that no later call starts from a stale count
  const size_t clear = (v & LILY_STATUS_TIMEOUT) ? 16 : 4;
  if (v && cudaMemsetAsync(ws_status(ws), 0, clear, s) != cudaSuccess) return LILY_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return LILY_ERR_CUDA;
  return (int)v;
}

uint64_t lily_moe_set_route_wait_ns(uint64_t ns) {
  return g_route_wait_ns.exchange(ns);
}

const char* lily_moe_strerror(int code) {
  switch (code) {
    case LILY_OK: return "ok";
    case LILY_ERR_INVALID_ARG: return "invalid argument";
    case LILY_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case LILY_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case LILY_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case LILY_ERR_ARCH: return "device is not compute capability 10.3 (sm_103a)";
    case LILY_ERR_CUDA: return "CUDA runtime error";
    case LILY_ERR_DEVICE: return "device status bits set";
    default: return "unknown error";
  }
}

int lily_moe_profile_enable(int enable) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = enable != 0;
  return LILY_OK;
}

int lily_moe_profile_read(double* total_ms, int64_t* launches) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (total_ms)
    for (int i = 0; i < LILY_KERNEL_KINDS; ++i) total_ms[i] = 0.0;
  if (launches)
    for (int i = 0; i < LILY_KERNEL_KINDS; ++i) launches[i] = 0;
  int rc = LILY_OK;
  for (auto& rec : g_prof_open) {
    float ms = 0.f;
    if (cudaEventSynchronize(rec.b) != cudaSuccess ||
        cudaEventElapsedTime(&ms, rec.a, rec.b) != cudaSuccess) {
      rc = LILY_ERR_CUDA;
      cudaGetLastError();  // do not leave this failure for the next call to find
    }
    if (rec.kind >= 0 && rec.kind < LILY_KERNEL_KINDS) {
      if (total_ms) total_ms[rec.kind] += ms;
      if (launches) launches[rec.kind] += 1;
    }
    g_prof_pool.push_back(rec.a);
    g_prof_pool.push_back(rec.b);
  }
  g_prof_open.clear();
  return rc;
}

const char* lily_moe_kernel_name(int kind) {
  static const char* names[] = {"router_gemm", "dec_router", "route", "gateup_gemm",
                                "down_gemm",   "combine",    "dec_gateup", "dec_down",
                                "unused",      "rmsnorm",     "unused", "unused",
                                "router_prep", "router_reduce", "token_rows"};
  if (kind < 0 || kind >= (int)(sizeof(names) / sizeof(names[0]))) return "unused";
  return names[kind];
}

const char* lily_moe_version(void) { return "lily_moe 0.1 sm_103a"; }

}  // extern "C"
