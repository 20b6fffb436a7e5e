// lily_internal.h -- host-side launchers shared by the library's translation
// units (not part of the public ABI).
#pragma once
#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/lily_moe.h"

namespace lily {

// Kernel kinds for the optional per-kernel event timing.
enum KernelKind : int {
  K_ROUTER_GEMM = 0,
  K_ROUTER_GEMV = 1,  // the decode router
  K_ROUTE = 2,
  K_GATEUP = 3,
  K_DOWN = 4,
  K_FINALIZE = 5,     // the combine of each token's output rows
  K_DEC_GATEUP = 6,
  K_DEC_DOWN = 7,
  K_RMSNORM = 9,
  K_ROUTER_PREP = 12,
  K_ROUTER_REDUCE = 13,
  K_TOKEN_ROWS = 14,
  K_NUM = 15
};

// Raise a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device; remembered, so the runtime call happens once per kernel,
// device and size (api.cu).
cudaError_t ensure_smem_attr(const void* func, size_t bytes);

// Profiling hooks (api.cu): bracket one launch with events when enabled.
void prof_begin(int kind, cudaStream_t s);
void prof_end(int kind, cudaStream_t s);

// Tokens handled by one block of the routing kernel.
constexpr int kRouteTok = 32;  // tokens per routing block, at most
// Tokens per routing block: 16 (two per warp) up to T = 2048, where the
// block-parallel top-k is the routing kernel's longest phase and SMs are
// idle, else 32 (more blocks would lengthen the histogram sums).
__host__ __device__ inline int route_tok(int T) { return T <= 2048 ? 16 : 32; }
__host__ __device__ inline int route_blocks(int T) { return (T + route_tok(T) - 1) / route_tok(T); }
constexpr int kRouteThreads = 256;

// Launch with the programmatic stream-serialization attribute (the kernel
// calls pdl_wait() before reading what its predecessor wrote).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------- routing
struct RouteArgs {
  const float* logits_src;  // fp32 [T][E]
  float* logits_dst;        // fp32 [T][E] (may equal logits_src)
  int T, E, k, BM, cap;
  int32_t* ids;
  float* gates;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv;
  int32_t* block_map;
  int32_t* n_tiles;
  int32_t* hist;       // workspace [nblk][E]
  uint32_t* bar;       // workspace: grid barrier {count, generation}
  uint32_t* status;    // workspace status word
  uint64_t wait_ns;    // give-up limit of the grid barrier's wait (route_wait_limit_ns())
};
// Current give-up limit of the routing kernel's grid-barrier wait (api.cu):
// 2 s unless lily_moe_set_route_wait_ns() changed it.
uint64_t route_wait_limit_ns();
// Decode router (T <= 8): logits only, plus x in the decode GEMV's B-fragment
// order (xpg, [T][d/64][32] words) with its 64-group sums (xsg, [T][d/64]).
// With `norm` x is the fp32 residual [T][d] of a layer stack and the scored
// rows are bf16(rmsnorm(x, eps)); else x is bf16 [T][d].
// Its last CTA to finish also routes the tokens: the routing outputs (route)
// and the step's tile slots (plan: slot count, then the slots) for the GEMVs.
struct DecRouterArgs {
  const void* x;
  const float* w;   // [E][d]
  const float* b;   // [E] or NULL
  float* logits;    // [T][E]
  uint32_t* xpg;
  float* xsg;
  float eps;
  int T, d, E;
  RouteArgs route;
  void* plan;       // decode plan (decode_plan_bytes())
  uint32_t* done;   // zero-initialised counter of finished CTAs, returned to zero
  // the experts' weights ([E+1] experts, d_ff F), prefetched into L2 as soon
  // as the step's experts are known (the shared expert at the start); F = 0:
  // no prefetch (expert pointers not given)
  int F;
  const uint8_t* gq; const uint16_t* gs; const uint16_t* gb;
  const uint8_t* uq; const uint16_t* us; const uint16_t* ub;
  const uint8_t* dq; const uint16_t* ds; const uint16_t* db;
};
size_t decode_plan_bytes();
cudaError_t launch_dec_router(const DecRouterArgs& a, bool norm, cudaStream_t s);
// Router on tensor cores for larger T: W split exactly into three bf16 terms
// (w_split, [3][E][d]), fp32 partial logits per K-split (partial,
// [router_splits(T,d)][T][E]) summed in order into logits (+ bias).
int router_splits(int T, int d);
size_t router_tc_smem(int E);
// w_presplit: the same split made ahead by launch_router_split, or NULL.
cudaError_t launch_router_tc(const void* x, const float* w, const float* bias, int T, int d,
                             int E, void* w_split, const void* w_presplit, float* partial,
                             float* logits, uint32_t* status, cudaStream_t s);
cudaError_t launch_router_split(const float* w, int E, int d, void* w_split, cudaStream_t s);
cudaError_t launch_route(const RouteArgs& a, cudaStream_t s);
int route_max_blocks();  // co-resident blocks of the routing kernel (0 = unknown)

// ---------------------------------------------------------------- prefill GEMMs
struct GemmArgs {
  int T, E, k, d, F, BM;
  const int32_t* block_map;
  const int32_t* n_tiles;
  const int32_t* offsets;
  const int32_t* perm;
  const float* gates;
  const uint16_t* s0;  // gate (or down) scales
  const uint16_t* b0;
  const uint16_t* s1;  // up scales (gate/up only)
  const uint16_t* b1;
  const int32_t* inv;  // inv_perm [P]: the expert-sorted row of pair t*k + j
  void* H;             // fp16 [P+T][F], 8-element chunks in K-chunk order, rows
                       // weighted by their gate
  void* O;             // fp16 [P+T][d] down GEMM output rows (gate applied), same order
  int4* tiles;         // [tile_count(T, E, k, BM)] {expert, row0, rows, 0}: shared-expert
                       // tiles first, then the block map's; rows = 0 marks no tile
  uint32_t* status;
};
// Tiles of the grouped GEMMs: ceil(T / BM) shared-expert tiles plus the block
// map's capacity.
__host__ __device__ inline int tile_count(int T, int E, int k, int BM) {
  const int P = T * k;
  return (T + BM - 1) / BM + (P + BM - 1) / BM + (E < P ? E : P);
}
// Token rows for the gate/up GEMM: xs[r] = fp16(x[perm[r] / k]) for the P
// expert-sorted rows and x16[t] = fp16(x[t]), every 8-element chunk in
// K-chunk order; the same launch writes the tile table a.tiles.  Then the
// gate/up GEMM (tensor maps built from the pointers), the down GEMM (output
// rows into a.O) and the combine of each token's rows.
cudaError_t launch_token_rows(const GemmArgs& a, const void* x, void* xs, void* x16, cudaStream_t s);
cudaError_t launch_gateup(const GemmArgs& a, const void* xs, const void* x16, const uint8_t* gq,
                          const uint8_t* uq, cudaStream_t s);
cudaError_t launch_down(const GemmArgs& a, const uint8_t* dq, cudaStream_t s);
// y[t] = sum of token t's rows of O (routed rows in slot order, then the
// shared row), fp32 (y_f32) or bf16; or, with x non-NULL, x[t] += that sum and
// xn[t] = bf16(rmsnorm(x[t], eps)) when xn is non-NULL.
cudaError_t launch_combine(const GemmArgs& a, void* y, bool y_f32, float* x, void* xn, float eps,
                           cudaStream_t s);
size_t gemm_smem_bytes(bool gateup, int BM, int K, int sub);
// Pipeline stages of a grouped GEMM (nout: its output features per matrix).
int gemm_stages(bool gateup, int BM, int K, int nout);

// ---------------------------------------------------------------- decode
// The decode GEMVs (T <= 8) read the step's tile slots from the plan the
// router launch wrote.
struct DecodeArgs {
  int T, E, k, d, F, BM, cap;
  const void* plan;     // the decode plan written by the router launch
  const uint8_t* gq; const uint16_t* gs; const uint16_t* gb;
  const uint8_t* uq; const uint16_t* us; const uint16_t* ub;
  const uint8_t* dq; const uint16_t* ds; const uint16_t* db;
  const uint32_t* xpg;  // x in B-fragment pair order [T][d/64][32] (router launch)
  const float* xsg;     // x 64-group sums [T][d/64]
  void* H;         // fp16 [P+T][F], each 64-group in the mma pair order
  void* y;         // [T][d], fp32 if y_f32 else bf16
  bool y_f32;
  float* resid;    // non-NULL: x_resid[t][:] += layer output (fp32), y unused (stacked decode)
  uint32_t* status;
};
// The two decode GEMV launches (gate/up + SwiGLU, down + combine), chained
// with programmatic dependent launch after the decode router.
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);

// ---------------------------------------------------------------- misc
cudaError_t launch_rmsnorm(const float* x, void* out, int T, int d, float eps, cudaStream_t s);


// Driver entry point for cuTensorMapEncodeTiled (resolved through the runtime).
CUresult encode_tiled(CUtensorMap* tm, CUtensorMapDataType dt, uint32_t rank, void* base,
                      const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                      CUtensorMapSwizzle swz);

}  // namespace lily
