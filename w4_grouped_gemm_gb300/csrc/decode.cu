// decode.cu -- W4 GEMV path for batch-1 / small-batch decode (1..8 rows).
//
// Batch-1 decode is bandwidth-bound, so the aim is every weight byte in
// flight as early as possible and the fewest instructions per weight byte
// (page "Lily Beats MLX-LM 1.35x on Decode: Perplexity's Rust+Metal Engine
// for Apple Silicon", section "Decode: eliminating per-token CPU round trips";
// verify batches of two to five rows are the speculative-decoding shapes of
// the same section).  Each distinct active expert (block-map tile) is
// streamed once for all its rows.
//
// Data movement: a work unit is 16 weight rows of one expert (the mma M).
// Its packed codes arrive by TMA in boxes of 16 rows x 128 bytes (64 bytes
// for 64-byte rows) with the matching 128- (64-) byte swizzle, so the mma
// fragment loads of eight rows at one K offset hit eight different bank
// groups; its scales and biases arrive by plain bulk copies.  One producer
// lane per CTA issues the copies of a ring of stages far ahead; eight
// consumer warps compute.
//
// Arithmetic per 64-weight group g of a row (w = s*q + b):
//   sum_k w_k x_k = s * (sum_k (q_k + c) x_k - c * X_g) + b * X_g,
//   X_g = sum_{k in g} x_k.
// The bracket runs on the tensor cores (mma.sync m16n8k16, fp32 accumulate):
// q + c is exact in the operand type and is made from the packed codes with
// one LOP3 per pair, so the weights are never rounded and no per-weight
// scale/bias arithmetic is needed.  Gate/up multiply bf16 x (c = 128, the
// bf16 magic); down multiplies the fp16 H (c = 1024, the fp16 magic).  The
// pairs come out as (q_i, q_{i+4}) of each 8-code word; the activations are
// laid out in that same order (x by the decode router; H by the gate/up
// kernel), so the K order of both operands agrees.
#include "routing.cuh"

namespace lily {

constexpr int kDecMaxRows = 8;        // mma N: token rows of one slot
constexpr int kDecUnitRows = 16;      // weight rows of one work unit (mma M)
constexpr int kDecConsumers = 8;      // consumer warps
constexpr int kDecThreads = 32 * (1 + kDecConsumers);  // warp 0: producer
// Two CTAs per SM by registers: a down CTA fits beside a gate/up CTA, so it
// can start streaming its weights while the gate/up kernel finishes.
constexpr int kDecMinBlocks = 2;
constexpr size_t kGuSmemBudget = 170 * 1024;  // gate/up: stages, partials, x, routing
constexpr size_t kDnStageBudget = 50 * 1024;  // down: weight stages
constexpr int kGuMaxStages = 4;
constexpr int kDnMaxStages = 16;

template <bool F16>
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  if (F16)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// (q_i + c, q_{i+4} + c) as a 16-bit float pair, i = 0..3, from one 8-code
// word: c = 128 with the bf16 magic 0x4300, c = 1024 with the fp16 magic 0x6400.
template <bool F16>
__device__ __forceinline__ void code_pairs(uint32_t w, uint32_t (&p)[4]) {
  const uint32_t magic = F16 ? 0x64006400u : 0x43004300u;
  p[0] = lop3_and_or(w, 0x000F000Fu, magic);
  p[1] = lop3_and_or(w >> 4, 0x000F000Fu, magic);
  p[2] = lop3_and_or(w >> 8, 0x000F000Fu, magic);
  p[3] = lop3_and_or(w >> 12, 0x000F000Fu, magic);
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t h) {
  return __uint_as_float((uint32_t)h << 16);
}

// Position of element j (0..63) of a 64-group in the pair order used for H:
// 16-bit index 2*word + half, word = c*8 + w*4 + (e & 3), half = e >> 2, for
// j = c*16 + 8w + e.  Word `word` of a group holds the (i, i+4) pair that one
// mma B-fragment register takes, so the down GEMV reads its fragments with
// plain 16-byte loads.
__host__ __device__ __forceinline__ int hpair_pos(int j) {
  const int c = j >> 4, w = (j >> 3) & 1, e = j & 7;
  return 2 * (c * 8 + w * 4 + (e & 3)) + (e >> 2);
}

// ---------------------------------------------------------------- layout
// Codes of a 16-row unit: row_bytes / rb boxes of [16 rows][rb bytes], rb =
// min(row_bytes, 128), with the TMA swizzle of that width: the 16-byte chunk
// index of row r is XOR-ed with (r & 7) for 128-byte rows and ((r >> 1) & 3)
// for 64-byte rows.
__host__ __device__ __forceinline__ int box_bytes(int row_bytes) {
  return row_bytes < 128 ? row_bytes : 128;
}
// Shared-memory offset of byte `off` of row r (0..15) of a unit whose boxes
// have rows of 1 << rbs bytes (64 or 128): shifts and masks only.
__device__ __forceinline__ uint32_t unit_off(int r, int off, int rbs) {
  const int box = off >> rbs, b = off & ((1 << rbs) - 1);
  const int phase = rbs == 7 ? (r & 7) : ((r >> 1) & 3);
  return (uint32_t)(((box * kDecUnitRows + r) << rbs) + ((((b >> 4) ^ phase)) << 4) + (b & 15));
}
__host__ __device__ __forceinline__ uint32_t round1k(uint32_t v) { return (v + 1023u) & ~1023u; }
// Gate/up stage: gate codes, up codes (16 rows x d/2 bytes each), then the
// gate scales, gate biases, up scales, up biases (16 rows x d/64 bf16 each).
__host__ __device__ __forceinline__ uint32_t gu_stage_bytes(int d) {
  return round1k((uint32_t)(2 * kDecUnitRows * (d / 2) + 4 * kDecUnitRows * (d / 64) * 2));
}
// Down stage: codes (16 rows x F/2 bytes), scales, biases (16 rows x F/64 bf16).
__host__ __device__ __forceinline__ uint32_t dn_stage_bytes(int F) {
  return round1k((uint32_t)(kDecUnitRows * (F / 2) + 2 * kDecUnitRows * (F / 64) * 2));
}
constexpr uint32_t kGuPartBytes = 2 * kDecConsumers * 2 * kDecUnitRows * kDecMaxRows * 4;
constexpr uint32_t kDnTileBytes = kDecConsumers * kDecMaxRows * kDecUnitRows * 4;
constexpr uint32_t kBarBytes = 512;  // mbarriers and flags

// One 64-group of 16 weight rows against B fragments xw (this lane's 8
// words: the (i, i+4) pairs of its K values for B column gi) and the group
// sums x0, x1 of accumulator columns 2c, 2c+1.  wa / wb: the lane's 16 codes
// of rows gi and gi+8; sa, ba, sb, bb: those rows' scale and bias.
template <bool F16>
__device__ __forceinline__ void group_mma(uint2 wa, uint2 wb, float sa, float ba, float sb,
                                          float bb, const uint32_t (&xw)[8], float x0, float x1,
                                          float (&out)[4]) {
  // four independent accumulators (one per k16 step): the four MMAs do not
  // wait for each other; their sums are added afterwards
  float part[4][4] = {};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t pa[4], pb[4];
    code_pairs<F16>(h == 0 ? wa.x : wa.y, pa);
    code_pairs<F16>(h == 0 ? wb.x : wb.y, pb);
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const uint32_t afrag[4] = {pa[2 * m], pb[2 * m], pa[2 * m + 1], pb[2 * m + 1]};
      mma_16816<F16>(part[h * 2 + m], afrag, xw[h * 4 + m * 2], xw[h * 4 + m * 2 + 1]);
    }
  }
  float acc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = (part[0][i] + part[1][i]) + (part[2][i] + part[3][i]);
  constexpr float off = F16 ? 1024.f : 128.f;  // the code offset of the magic
  out[0] += sa * (acc[0] - off * x0) + ba * x0;
  out[1] += sa * (acc[1] - off * x1) + ba * x1;
  out[2] += sb * (acc[2] - off * x0) + bb * x0;
  out[3] += sb * (acc[3] - off * x1) + bb * x1;
}

// Codes of rows gi and gi+8 for this lane's 16 K values of group g.
__device__ __forceinline__ void unit_codes(const uint8_t* unit, int g, int gi, int c, int rbs,
                                           uint2& wa, uint2& wb) {
  const int off = g * 32 + c * 8;
  wa = *reinterpret_cast<const uint2*>(unit + unit_off(gi, off, rbs));
  wb = *reinterpret_cast<const uint2*>(unit + unit_off(gi + 8, off, rbs));
}


// Give-up flag shared by the roles of a CTA (see mbar_wait).
struct DecFlags {
  int abort;
};

// The plan (written by the router launch, complete once this grid may read
// it) into shared memory: every slot is loaded in parallel with the count,
// one round trip; returns the count (valid after the next __syncthreads).
__device__ __forceinline__ int load_plan(const void* plan, DecSlot* slots, int* nslots_s) {
  const DecPlan* p = static_cast<const DecPlan*>(plan);
  constexpr int kWords = kMaxSlots * (int)sizeof(DecSlot) / 16;
  const int4* src = reinterpret_cast<const int4*>(p->slot);
  for (int i = threadIdx.x; i < kWords; i += blockDim.x)
    reinterpret_cast<int4*>(slots)[i] = __ldcg(src + i);
  if (threadIdx.x == 0) *nslots_s = min(max(__ldcg(&p->nslots), 1), kMaxSlots);
  __syncthreads();
  return *nslots_s;
}

// The slot plan, x in fragment order (nx 16-byte words) and the group sums
// (nxs floats) into shared memory, with up to four words per thread in flight
// before their stores (one round trip for the lot instead of one per array).
__device__ __forceinline__ int load_plan_x(const void* plan, DecSlot* slots, int* nslots_s,
                                           const uint4* xpg, uint4* xpg_s, int nx,
                                           const float* xsg, float* xsg_s, int nxs) {
  const DecPlan* p = static_cast<const DecPlan*>(plan);
  constexpr int kWords = kMaxSlots * (int)sizeof(DecSlot) / 16;
  const int4* src = reinterpret_cast<const int4*>(p->slot);
  const int n = kWords + nx, nt = blockDim.x, tid = threadIdx.x;
  for (int base = 0; base < n; base += 4 * nt) {
    int4 v[4];
    float xs = 0.f;
    int ns = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = base + u * nt + tid;
      if (i < kWords)
        v[u] = __ldcg(src + i);
      else if (i < n)
        v[u] = __ldcg(reinterpret_cast<const int4*>(xpg) + (i - kWords));
    }
    if (base == 0) {
      if (tid < nxs) xs = __ldcg(xsg + tid);
      if (tid == 0) ns = __ldcg(&p->nslots);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = base + u * nt + tid;
      if (i < kWords)
        reinterpret_cast<int4*>(slots)[i] = v[u];
      else if (i < n)
        reinterpret_cast<int4*>(xpg_s)[i - kWords] = v[u];
    }
    if (base == 0) {
      if (tid < nxs) xsg_s[tid] = xs;
      if (tid == 0) *nslots_s = min(max(ns, 1), kMaxSlots);
    }
  }
  for (int i = tid + nt; i < nxs; i += nt) xsg_s[i] = __ldcg(xsg + i);
  __syncthreads();
  return *nslots_s;
}

// ======================================================= decode router
// Logits of T <= 8 rows: CTA b scores experts 2b and 2b+1, four warps per
// expert, each over a quarter of d, with its quarter of the weight row
// loaded into registers before the wait for the predecessor (the weights are
// static); the four quarter sums are added in a fixed order.  The same launch
// writes x in the expert GEMV's B-fragment order with its 64-group sums:
//   xpg[(t*G + g)*32 + c*8 + w*4 + e] = (x[t][g*64 + c*16 + 8w + e], x[...+4])
//   xsg[t*G + g] = sum of x[t][g*64 .. g*64+63]
// With NORM the input is the fp32 residual of a layer stack and the scored
// rows are bf16(x / sqrt(mean(x^2) + eps)) (unit-weight RMSNorm).
constexpr int kDecRouterThreads = 256;
constexpr int kDecRouterEpb = 2;     // experts per CTA
constexpr int kDecRouterWv = 8;      // float4 of a quarter row per lane: d <= 4096

// Part `part` of `nparts` of expert e's weights (its nine arrays) into L2,
// one bulk prefetch per array (32-bit sizes: one matrix is at most 8 MB).
__device__ __forceinline__ void prefetch_expert(const DecRouterArgs& a, int e, int part,
                                                int nparts) {
  const uint32_t n = (uint32_t)a.F * (uint32_t)a.d;  // weights of one matrix
  const size_t eo = (size_t)e * n;
  const void* base[9] = {a.gq + eo / 2, a.uq + eo / 2, a.dq + eo / 2,
                         a.gs + eo / 64, a.gb + eo / 64, a.us + eo / 64,
                         a.ub + eo / 64, a.ds + eo / 64, a.db + eo / 64};
#pragma unroll
  for (int r = 0; r < 9; ++r) {
    const uint32_t bytes = r < 3 ? n / 2 : n / 32;
    const uint32_t chunk = ((bytes + (uint32_t)nparts - 1) / (uint32_t)nparts + 15u) & ~15u;
    const uint32_t off = (uint32_t)part * chunk;
    if (off < bytes)
      prefetch_l2(static_cast<const uint8_t*>(base[r]) + off, min(chunk, bytes - off));
  }
}

template <bool NORM>
__global__ void __launch_bounds__(kDecRouterThreads) dec_router_kernel(const DecRouterArgs a) {
  __shared__ float s_part[kDecRouterEpb][4][kDecMaxRows];
  __shared__ float s_red[kDecRouterThreads / 32][kDecMaxRows];
  __shared__ float s_inv[kDecMaxRows];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = a.T, d = a.d, E = a.E;
  const int el = warp >> 2, qd = warp & 3;
  const int e = blockIdx.x * kDecRouterEpb + el;
  const bool has = e < E;
  const int nq4 = d / 16;  // float4 in a quarter row
  const float4* wq = reinterpret_cast<const float4*>(a.w + (size_t)(has ? e : 0) * d) + qd * nq4;
  // the shared expert serves every token: its weights head for L2 at once
  if (a.F > 0 && threadIdx.x == 0) prefetch_expert(a, E, blockIdx.x, gridDim.x);
  float4 wv[kDecRouterWv];
#pragma unroll
  for (int i = 0; i < kDecRouterWv; ++i) {  // static: before the wait
    const int f = i * 32 + lane;
    wv[i] = (has && f < nq4) ? __ldg(wq + f) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  pdl_wait();  // x comes from the predecessor
  pdl_trigger();
  if (NORM) {
    const float* xr = static_cast<const float*>(a.x);
    for (int t = 0; t < T; ++t) {
      float ss = 0.f;
      for (int i = threadIdx.x * 4; i < d; i += kDecRouterThreads * 4) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(xr + (size_t)t * d + i));
        ss = fmaf(v.x, v.x, ss);
        ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss);
        ss = fmaf(v.w, v.w, ss);
      }
      ss = warp_sum(ss);
      if (lane == 0) s_red[warp][t] = ss;
    }
    __syncthreads();
    if (threadIdx.x < T) {
      float tot = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < kDecRouterThreads / 32; ++w2) tot += s_red[w2][threadIdx.x];
      s_inv[threadIdx.x] = 1.f / sqrtf(tot / (float)d + a.eps);
    }
    __syncthreads();
  }
  // element i of row t as scored: exact bf16 values
  auto xval4 = [&](int t, int i) {  // i a multiple of 4
    if (NORM) {
      const float4 v = __ldcg(
          reinterpret_cast<const float4*>(static_cast<const float*>(a.x) + (size_t)t * d + i));
      const float s = s_inv[t];
      return make_float4(__bfloat162float(__float2bfloat16_rn(v.x * s)),
                         __bfloat162float(__float2bfloat16_rn(v.y * s)),
                         __bfloat162float(__float2bfloat16_rn(v.z * s)),
                         __bfloat162float(__float2bfloat16_rn(v.w * s)));
    }
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(
        static_cast<const uint16_t*>(a.x) + (size_t)t * d + i));
    return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u),
                       __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u));
  };
  float acc[kDecMaxRows];
#pragma unroll
  for (int t = 0; t < kDecMaxRows; ++t) acc[t] = 0.f;
#pragma unroll
  for (int i = 0; i < kDecRouterWv; ++i) {
    const int f = i * 32 + lane;
    if (f < nq4) {
#pragma unroll
      for (int t = 0; t < kDecMaxRows; ++t) {
        if (t < T) {
          const float4 x4 = xval4(t, (qd * nq4 + f) * 4);
          acc[t] = fmaf(wv[i].x, x4.x, acc[t]);
          acc[t] = fmaf(wv[i].y, x4.y, acc[t]);
          acc[t] = fmaf(wv[i].z, x4.z, acc[t]);
          acc[t] = fmaf(wv[i].w, x4.w, acc[t]);
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kDecMaxRows; ++t) {
    const float v = warp_sum(acc[t]);
    if (lane == 0 && t < T) s_part[el][qd][t] = v;
  }
  __syncthreads();
  if (threadIdx.x < kDecRouterEpb * T) {
    const int el2 = threadIdx.x / T, t = threadIdx.x % T, e2 = blockIdx.x * kDecRouterEpb + el2;
    if (e2 < E) {
      float v = s_part[el2][0][t];
      v += s_part[el2][1][t];
      v += s_part[el2][2][t];
      v += s_part[el2][3][t];
      a.logits[(size_t)t * E + e2] = v + (a.b ? __ldg(a.b + e2) : 0.f);
    }
  }
  // x in the expert GEMV's fragment order, with its group sums
  const int G = d / 64;
  for (int u = blockIdx.x * (kDecRouterThreads / 32) + warp; u < T * G;
       u += gridDim.x * (kDecRouterThreads / 32)) {
    const int t = u / G, g = u % G;
    const int c = lane >> 3, w2 = (lane >> 2) & 1, e4 = lane & 3;
    const int i = g * 64 + c * 16 + 8 * w2 + e4;
    float lo, hi;
    if (NORM) {
      const float* xr = static_cast<const float*>(a.x) + (size_t)t * d;
      lo = __bfloat162float(__float2bfloat16_rn(__ldcg(xr + i) * s_inv[t]));
      hi = __bfloat162float(__float2bfloat16_rn(__ldcg(xr + i + 4) * s_inv[t]));
    } else {
      const uint16_t* xh = static_cast<const uint16_t*>(a.x) + (size_t)t * d;
      lo = __uint_as_float((uint32_t)xh[i] << 16);
      hi = __uint_as_float((uint32_t)xh[i + 4] << 16);
    }
    a.xpg[(size_t)u * 32 + lane] = (__float_as_uint(lo) >> 16) | (__float_as_uint(hi) & 0xFFFF0000u);
    const float sum = warp_sum(lo + hi);
    if (lane == 0) a.xsg[u] = sum;
  }
  // the CTA that finishes last routes: every CTA counts itself done with one
  // acquire-release add (after the CTA barrier, so it orders every write of
  // the CTA before it, and the last CTA's reads of the logits after it)
  __shared__ int s_last;
  __shared__ __align__(16) float s_lg[kDecMaxRows * kMaxE];
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(a.done) : "memory");
    s_last = old == gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return;
  for (int i = threadIdx.x; i < T * E; i += kDecRouterThreads) s_lg[i] = __ldcg(a.logits + i);
  __syncthreads();
  DecPlan* plan = static_cast<DecPlan*>(a.plan);
  small_routing(s_lg, T, E, a.route.k, a.route.BM, plan->slot, &plan->nslots, &a.route,
                a.route.status);
  if (threadIdx.x == 0) *a.done = 0;  // back to zero for the next call
}

size_t decode_plan_bytes() { return sizeof(DecPlan); }

// Shared memory as large as it goes on every SM that runs a decode kernel, so
// that a CTA of the next kernel in the chain fits beside one of the current
// kernel (an SM's L1/shared split is fixed while CTAs run on it).
static void carveout_max(const void* kern) {
  cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                       (int)cudaSharedmemCarveoutMaxShared);
}

cudaError_t launch_dec_router(const DecRouterArgs& a, bool norm, cudaStream_t s) {
  if (a.T < 1 || a.T > kDecMaxRows || a.d % 128 || a.d / 16 > 32 * kDecRouterWv || a.E > 256)
    return cudaErrorInvalidValue;
  const int grid = (a.E + kDecRouterEpb - 1) / kDecRouterEpb;
  static bool attr_set = false;  // (idempotent: races only repeat the call)
  if (!attr_set) {
    carveout_max((const void*)dec_router_kernel<true>);
    carveout_max((const void*)dec_router_kernel<false>);
    attr_set = true;
  }
  prof_begin(K_ROUTER_GEMV, s);
  const cudaError_t err =
      norm ? launch_pdl(dec_router_kernel<true>, dim3(grid), dim3(kDecRouterThreads), 0, s, a)
           : launch_pdl(dec_router_kernel<false>, dim3(grid), dim3(kDecRouterThreads), 0, s, a);
  prof_end(K_ROUTER_GEMV, s);
  return err;
}

// Shared-memory regions of the GEMV kernels after their weight stages.
struct DecSmem {
  uint32_t lg, slots, xpg, xsg, part, bars, total;
};
// gate/up: logits, slots, x fragments and sums, partial sums, barriers
__host__ __device__ inline DecSmem gu_smem(int T, int E, int d, int nstages) {
  DecSmem m;
  const int G = d / 64;
  uint32_t off = 1024 + (uint32_t)nstages * gu_stage_bytes(d);  // alignment slack + stages
  m.lg = 0;
  m.slots = off; off += (uint32_t)kMaxSlots * sizeof(DecSlot);
  m.xpg = off;   off += (uint32_t)T * G * 128;
  m.xsg = off;   off += (uint32_t)(T * G * 4 + 15) & ~15u;
  m.part = off;  off += kGuPartBytes;
  m.bars = off;  off += kBarBytes;
  m.total = off;
  return m;
}
// down: logits, slots, per-warp output tiles, barriers
__host__ __device__ inline DecSmem dn_smem(int T, int E, int F, int nstages) {
  DecSmem m;
  uint32_t off = 1024 + (uint32_t)nstages * dn_stage_bytes(F);
  m.lg = 0;
  m.slots = off; off += (uint32_t)kMaxSlots * sizeof(DecSlot);
  m.xpg = m.xsg = 0;
  m.part = off;  off += kDnTileBytes;
  m.bars = off;  off += kBarBytes;
  m.total = off;
  return m;
}

// ======================================================= gate/up + SwiGLU
// Work item = (tile slot, 16 rows of F) for both matrices; item i runs on
// CTA i % grid.  The first item of CTAs 0 .. F/16-1 belongs to the shared
// expert (slot 0), which needs no routing: its weights are requested before
// the wait for the router.  Then every CTA loads the slot plan (written by
// the router's last CTA) and the x fragments, and streams its items'
// weights through a ring of stages, one 3-D copy per matrix and item.
// Per item each consumer warp takes the groups g = warp, warp + 8, ... of
// both matrices; the eight partial 16 x 8 results are summed in a fixed order
// and H = silu(g) * u is written as fp16 in the pair order the down GEMV reads.
__global__ void __launch_bounds__(kDecThreads, kDecMinBlocks)
    dec_gateup_kernel(const __grid_constant__ CUtensorMap tm_g,
                      const __grid_constant__ CUtensorMap tm_u, const DecodeArgs a,
                      const int nstages) {
  extern __shared__ uint8_t smem_raw[];
  // aligned up to 1024 bytes by pointer arithmetic on the shared array, so
  // the compiler keeps the accesses in the shared window (not generic)
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int T = a.T, d = a.d, F = a.F, G = d / 64;
  const int rb = box_bytes(d / 2), rbs = rb == 128 ? 7 : 6;
  const uint32_t SB = gu_stage_bytes(d);
  const uint32_t code_bytes = kDecUnitRows * (d / 2), sc_bytes = kDecUnitRows * G * 2;
  const DecSmem M = gu_smem(T, a.E, d, nstages);
  uint8_t* smem = base;  // stages at the start
  DecSlot* slots = (DecSlot*)(base + (M.slots - 1024));
  uint32_t* xpg_s = (uint32_t*)(base + (M.xpg - 1024));
  float* xsg_s = (float*)(base + (M.xsg - 1024));
  float* part = (float*)(base + (M.part - 1024));
  uint64_t* full = (uint64_t*)(base + (M.bars - 1024));
  uint64_t* empty = full + kGuMaxStages;
  uint64_t* cons = empty + kGuMaxStages;  // [2] consumer warps' hand-off
  DecFlags* fl = (DecFlags*)(cons + 2);
  int* nslots_s = (int*)(fl + 1);
  volatile int* abort = &fl->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nfb = F / kDecUnitRows;
  const int n_items = (1 + min(a.E, T * a.k)) * nfb;

  if (threadIdx.x == 0) {
    for (int i = 0; i < nstages; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    mbar_init(smem_u32(&cons[0]), kDecConsumers);
    mbar_init(smem_u32(&cons[1]), kDecConsumers);
    fl->abort = 0;
    fence_mbar_init();
    prefetch_tensormap(&tm_g);
    prefetch_tensormap(&tm_u);
  }
  __syncthreads();

  // the weights of item `it` (expert, 16-row block) into stage st
  auto issue = [&](int it, int expert, uint32_t st) {
    uint8_t* sp = smem + (size_t)st * SB;
    const uint32_t fb = smem_u32(&full[st]);
    mbar_arrive_expect_tx(fb, 2 * code_bytes + 4 * sc_bytes);
    const int row0 = expert * F + (it % nfb) * kDecUnitRows;
    tma_load_3d(smem_u32(sp), &tm_g, 0, row0, 0, fb);
    tma_load_3d(smem_u32(sp + code_bytes), &tm_u, 0, row0, 0, fb);
    const size_t so = (size_t)row0 * G;
    bulk_load(smem_u32(sp + 2 * code_bytes), a.gs + so, sc_bytes, fb);
    bulk_load(smem_u32(sp + 2 * code_bytes + sc_bytes), a.gb + so, sc_bytes, fb);
    bulk_load(smem_u32(sp + 2 * code_bytes + 2 * sc_bytes), a.us + so, sc_bytes, fb);
    bulk_load(smem_u32(sp + 2 * code_bytes + 3 * sc_bytes), a.ub + so, sc_bytes, fb);
  };
  // the shared expert's first item needs no routing: before the wait
  const bool early = (int)blockIdx.x < nfb;
  if (early && threadIdx.x == 0) issue(blockIdx.x, a.E, 0);

  pdl_wait();  // the plan and x fragments come from the router
  pdl_trigger();
  const int nslots = load_plan_x(a.plan, slots, nslots_s, reinterpret_cast<const uint4*>(a.xpg),
                                 reinterpret_cast<uint4*>(xpg_s), T * G * 8, a.xsg, xsg_s, T * G);

  if (warp == 0) {
    // ================================================= producer (warp 0)
    // this CTA's items with a slot: it = blockIdx.x + u * gridDim.x < nslots * nfb
    const int valid = nslots * nfb;
    const int nmine = valid > (int)blockIdx.x ? (valid - (int)blockIdx.x + (int)gridDim.x - 1) /
                                                    (int)gridDim.x
                                              : 0;
    const int first = nmine < nstages ? nmine : nstages;
    // the first round of the ring: lane u issues item u (in parallel)
    if (lane < first && !(early && lane == 0)) {
      const int it = blockIdx.x + lane * gridDim.x;
      issue(it, slots[it / nfb].expert, lane);
    }
    __syncwarp();
    if (lane == 0) {
      uint32_t u = first;
      for (; (int)u < nmine; ++u) {
        const int it = blockIdx.x + u * gridDim.x;
        const uint32_t st = u % nstages;
        if (!mbar_wait(smem_u32(&empty[st]), ((u / nstages) - 1) & 1, abort, a.status)) break;
        issue(it, slots[it / nfb].expert, st);
      }
      if (*abort) {  // let the copies in flight land before the CTA exits
        int never = 0;
        for (uint32_t k2 = (u > (uint32_t)nstages ? u - nstages : 0); k2 < u; ++k2)
          mbar_wait(smem_u32(&full[k2 % nstages]), (k2 / nstages) & 1, &never, a.status);
      }
    }
    return;
  }

  // =================================================== consumers (8 warps)
  const int cw = warp - 1, ct = threadIdx.x - 32;
  const int gi = lane >> 2, c = lane & 3;
  uint32_t u = 0;
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const int slot = it / nfb, fb = it % nfb;
    if (slot >= nslots) break;
    const DecSlot& sl = slots[slot];
    const uint32_t st = u % nstages;
    if (!warp_wait_all(smem_u32(&full[st]), (u / nstages) & 1, abort, a.status)) break;
    // B column gi: slot row gi (zero beyond the slot's rows); accumulator
    // columns 2c, 2c+1 take their rows' group sums
    const int rows = sl.rows;
    const int tg = sl.tok[min(gi, rows - 1)];
    const int t0 = sl.tok[min(2 * c, rows - 1)], t1 = sl.tok[min(2 * c + 1, rows - 1)];
    const uint32_t* xrow = xpg_s + (size_t)tg * G * 32 + c * 8;
    const uint8_t* sp = smem + (size_t)st * SB;
    const uint16_t* sc = reinterpret_cast<const uint16_t*>(sp + 2 * code_bytes);
    float og[4] = {0.f, 0.f, 0.f, 0.f}, ou[4] = {0.f, 0.f, 0.f, 0.f};
    for (int g = cw; g < G; g += kDecConsumers) {
      uint4 h0 = make_uint4(0, 0, 0, 0), h1 = h0;
      if (gi < rows) {
        h0 = *reinterpret_cast<const uint4*>(xrow + (size_t)g * 32);
        h1 = *reinterpret_cast<const uint4*>(xrow + (size_t)g * 32 + 4);
      }
      const uint32_t xw[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
      const float x0 = 2 * c < rows ? xsg_s[t0 * G + g] : 0.f;
      const float x1 = 2 * c + 1 < rows ? xsg_s[t1 * G + g] : 0.f;
      uint2 wa, wb;
      unit_codes(sp, g, gi, c, rbs, wa, wb);
      group_mma<false>(wa, wb, bf16_bits_to_float(sc[gi * G + g]),
                       bf16_bits_to_float(sc[kDecUnitRows * G + gi * G + g]),
                       bf16_bits_to_float(sc[(gi + 8) * G + g]),
                       bf16_bits_to_float(sc[kDecUnitRows * G + (gi + 8) * G + g]), xw, x0, x1, og);
      unit_codes(sp + code_bytes, g, gi, c, rbs, wa, wb);
      group_mma<false>(wa, wb, bf16_bits_to_float(sc[2 * kDecUnitRows * G + gi * G + g]),
                       bf16_bits_to_float(sc[3 * kDecUnitRows * G + gi * G + g]),
                       bf16_bits_to_float(sc[2 * kDecUnitRows * G + (gi + 8) * G + g]),
                       bf16_bits_to_float(sc[3 * kDecUnitRows * G + (gi + 8) * G + g]), xw, x0,
                       x1, ou);
    }
    float* pb = part + (size_t)(u & 1) * (kDecConsumers * 2 * kDecUnitRows * kDecMaxRows);
    float* pg = pb + (size_t)cw * 2 * kDecUnitRows * kDecMaxRows;
    float* pu = pg + kDecUnitRows * kDecMaxRows;
    pg[gi * 8 + 2 * c] = og[0];
    pg[gi * 8 + 2 * c + 1] = og[1];
    pg[(gi + 8) * 8 + 2 * c] = og[2];
    pg[(gi + 8) * 8 + 2 * c + 1] = og[3];
    pu[gi * 8 + 2 * c] = ou[0];
    pu[gi * 8 + 2 * c + 1] = ou[1];
    pu[(gi + 8) * 8 + 2 * c] = ou[2];
    pu[(gi + 8) * 8 + 2 * c + 1] = ou[3];
    // every consumer warp has read the stage and written its partials
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&cons[u & 1]));
    if (!warp_wait_all(smem_u32(&cons[u & 1]), (u >> 1) & 1, abort, a.status)) break;
    if (ct == 0) mbar_arrive(smem_u32(&empty[st]));
    if (ct < kDecUnitRows * kDecMaxRows) {
      const int row = ct >> 3, n = ct & 7;
      float gs = 0.f, us = 0.f;
#pragma unroll
      for (int w = 0; w < kDecConsumers; ++w) {
        gs += pb[(size_t)w * 2 * kDecUnitRows * kDecMaxRows + row * 8 + n];
        us += pb[(size_t)w * 2 * kDecUnitRows * kDecMaxRows + kDecUnitRows * kDecMaxRows +
                 row * 8 + n];
      }
      if (n < rows) {
        const float h = gs / (1.f + __expf(-gs)) * us;
        if (!(fabsf(h) <= 65504.f)) set_status(a.status, LILY_STATUS_F16_RANGE);
        const int f = fb * kDecUnitRows + row;  // H row in pair order, one 64-group after another
        static_cast<__half*>(a.H)[(size_t)(sl.row0 + n) * F + (f & ~63) + hpair_pos(f & 63)] =
            __float2half_rn(h);
      }
    }
    ++u;
  }
}

// ======================================================= down + combine
// CTA = 16 output features over every slot of the step.  Before waiting for
// the gate/up kernel the CTA routes the tokens itself from the logits (which
// the router wrote before the gate/up kernel could start, and this kernel
// starts only after every gate/up CTA has waited for the router) and its
// producer lane requests every slot's 16 weight rows, so the weights stream
// while the gate/up kernel runs.  Slot v goes to consumer warp v % 8, which
// runs the 16-row W4 GEMV over K = F against the slot's H rows (B fragments
// loaded from H; group sums from the same loads) and adds gate * out into its
// own [token][feature] tile.  The tiles are summed in warp order, so the
// result is deterministic.  The sum is written to y, or added to the fp32
// residual (stacked decode).
__global__ void __launch_bounds__(kDecThreads, kDecMinBlocks)
    dec_down_kernel(const __grid_constant__ CUtensorMap tm_d, const DecodeArgs a,
                    const int nstages) {
  extern __shared__ uint8_t smem_raw[];
  // aligned up to 1024 bytes by pointer arithmetic on the shared array, so
  // the compiler keeps the accesses in the shared window (not generic)
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int T = a.T, F = a.F, G = F / 64;
  const int rb = box_bytes(F / 2), rbs = rb == 128 ? 7 : 6;
  const uint32_t SB = dn_stage_bytes(F);
  const uint32_t code_bytes = kDecUnitRows * (F / 2), sc_bytes = kDecUnitRows * G * 2;
  const DecSmem M = dn_smem(T, a.E, F, nstages);
  uint8_t* smem = base;
  DecSlot* slots = (DecSlot*)(base + (M.slots - 1024));
  float* ytile = (float*)(base + (M.part - 1024));
  uint64_t* full = (uint64_t*)(base + (M.bars - 1024));
  uint64_t* empty = full + kDnMaxStages;
  uint64_t* done = empty + kDnMaxStages;
  DecFlags* fl = (DecFlags*)(done + 1);
  int* nslots_s = (int*)(fl + 1);
  volatile int* abort = &fl->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int f0 = blockIdx.x * kDecUnitRows;  // output features [f0, f0 + 16)

  if (threadIdx.x == 0) {
    for (int i = 0; i < nstages; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    mbar_init(smem_u32(done), kDecConsumers);
    fl->abort = 0;
    fence_mbar_init();
    prefetch_tensormap(&tm_d);
  }
  const int nslots = load_plan(a.plan, slots, nslots_s);  // before the wait: see above
  __syncthreads();

  if (warp == 0) {
    // the weights of slot v into stage st
    auto issue = [&](int v, uint32_t st) {
      uint8_t* sp = smem + (size_t)st * SB;
      const uint32_t fb = smem_u32(&full[st]);
      mbar_arrive_expect_tx(fb, code_bytes + 2 * sc_bytes);
      const int row0 = slots[v].expert * a.d + f0;
      tma_load_3d(smem_u32(sp), &tm_d, 0, row0, 0, fb);
      const size_t so = (size_t)row0 * G;
      bulk_load(smem_u32(sp + code_bytes), a.ds + so, sc_bytes, fb);
      bulk_load(smem_u32(sp + code_bytes + sc_bytes), a.db + so, sc_bytes, fb);
    };
    // the first round of the ring, before the wait: lane v issues slot v
    const int first = nslots < nstages ? nslots : nstages;
    if (lane < first) issue(lane, lane);
    __syncwarp();
    pdl_wait();
    pdl_trigger();
    if (lane == 0) {
      int v = first;
      for (; v < nslots; ++v) {
        const uint32_t st = v % nstages;
        if (!mbar_wait(smem_u32(&empty[st]), ((v / nstages) - 1) & 1, abort, a.status)) break;
        issue(v, st);
      }
      if (*abort) {
        int never = 0;
        for (int k2 = (v > nstages ? v - nstages : 0); k2 < v; ++k2)
          mbar_wait(smem_u32(&full[k2 % nstages]), (k2 / nstages) & 1, &never, a.status);
      }
    }
    return;
  }

  // =================================================== consumers (8 warps)
  pdl_wait();  // H comes from the gate/up kernel
  pdl_trigger();
  const int cw = warp - 1, ct = threadIdx.x - 32;
  const int gi = lane >> 2, c = lane & 3;
  float* yt = ytile + (size_t)cw * kDecMaxRows * kDecUnitRows;
  for (int i = lane; i < kDecMaxRows * kDecUnitRows; i += 32) yt[i] = 0.f;
  __syncwarp();
  const uint16_t* H = static_cast<const uint16_t*>(a.H);
  bool ok = true;
  for (int v = cw; v < nslots; v += kDecConsumers) {
    const DecSlot& sl = slots[v];
    const uint32_t st = v % nstages;
    if (!warp_wait_all(smem_u32(&full[st]), (v / nstages) & 1, abort, a.status)) {
      ok = false;
      break;
    }
    const int rows = sl.rows;
    // this lane's B column: slot row gi (zero beyond the slot's rows); the
    // slot's H fragments of every group loaded together
    const uint16_t* hrow = H + (size_t)(sl.row0 + min(gi, rows - 1)) * F + c * 16;
    const uint8_t* sp = smem + (size_t)st * SB;
    const uint16_t* sc = reinterpret_cast<const uint16_t*>(sp + code_bytes);
    float o[4] = {0.f, 0.f, 0.f, 0.f};
    // H fragments of two groups at a time, the next two requested before the
    // current two are used
    constexpr int kHc = 2;
    uint4 hh[kHc][2], hn[kHc][2];
    auto load_h = [&](int g0, uint4 (&dst)[kHc][2]) {
#pragma unroll
      for (int i = 0; i < kHc; ++i) {
        dst[i][0] = dst[i][1] = make_uint4(0, 0, 0, 0);
        if (g0 + i < G && gi < rows) {
          dst[i][0] = __ldcg(reinterpret_cast<const uint4*>(hrow + (g0 + i) * 64));
          dst[i][1] = __ldcg(reinterpret_cast<const uint4*>(hrow + (g0 + i) * 64 + 8));
        }
      }
    };
    load_h(0, hn);
    for (int g0 = 0; g0 < G; g0 += kHc) {
#pragma unroll
      for (int i = 0; i < kHc; ++i) {
        hh[i][0] = hn[i][0];
        hh[i][1] = hn[i][1];
      }
      if (g0 + kHc < G) load_h(g0 + kHc, hn);
#pragma unroll
      for (int i = 0; i < kHc; ++i) {
        const int g = g0 + i;
        if (g >= G) break;
        const uint32_t xw[8] = {hh[i][0].x, hh[i][0].y, hh[i][0].z, hh[i][0].w,
                                hh[i][1].x, hh[i][1].y, hh[i][1].z, hh[i][1].w};
        // X_g of slot row gi: this lane's 16 values, then over the 4 lanes c
        float xsum = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e)
          xsum += __half2float(__ushort_as_half((uint16_t)(xw[e] & 0xFFFFu))) +
                  __half2float(__ushort_as_half((uint16_t)(xw[e] >> 16)));
        xsum += __shfl_xor_sync(0xffffffffu, xsum, 1);
        xsum += __shfl_xor_sync(0xffffffffu, xsum, 2);
        // accumulator columns 2c, 2c+1 are slot rows 2c, 2c+1: their X_g
        const float x0 = __shfl_sync(0xffffffffu, xsum, (2 * c) * 4);
        const float x1 = __shfl_sync(0xffffffffu, xsum, (2 * c + 1) * 4);
        uint2 wa, wb;
        unit_codes(sp, g, gi, c, rbs, wa, wb);
        group_mma<true>(wa, wb, bf16_bits_to_float(sc[gi * G + g]),
                        bf16_bits_to_float(sc[kDecUnitRows * G + gi * G + g]),
                        bf16_bits_to_float(sc[(gi + 8) * G + g]),
                        bf16_bits_to_float(sc[kDecUnitRows * G + (gi + 8) * G + g]), xw, x0, x1,
                        o);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[st]));  // stage read
    // gate * out into this warp's tile: slot row n -> its token and gate
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int n = 2 * c + h;
      if (n < rows) {
        const int tok = sl.tok[n];
        const float gate = sl.gate[n];
        yt[tok * kDecUnitRows + gi] += gate * o[h];
        yt[tok * kDecUnitRows + gi + 8] += gate * o[2 + h];
      }
    }
  }
  if (!ok) return;
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_u32(done));
  if (!warp_wait_all(smem_u32(done), 0, abort, a.status)) return;
  for (int i = ct; i < T * kDecUnitRows; i += 32 * kDecConsumers) {
    const int t = i / kDecUnitRows, f = i % kDecUnitRows;
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < kDecConsumers; ++w) acc += ytile[(size_t)w * kDecMaxRows * kDecUnitRows + i];
    const size_t o = (size_t)t * a.d + f0 + f;
    if (a.resid)
      a.resid[o] += acc;
    else if (a.y_f32)
      static_cast<float*>(a.y)[o] = acc;
    else
      static_cast<__nv_bfloat16*>(a.y)[o] = __float2bfloat16_rn(acc);
  }
}

// ---------------------------------------------------------------- host side
// Packed codes of 16-row units as one copy: the rows of a unit cut into
// chunks of rb bytes (the swizzle span), chunk-major in shared memory (chunk
// b's 16 rows at b * 16 * rb), i.e. the layout of one 16 x rb box per chunk,
// with the same swizzle phase (row index mod 8), from a single 3-D copy:
// dimensions (byte within the chunk, row, chunk) with strides (row_bytes, rb).
static bool codes_map(CUtensorMap* tm, const uint8_t* q, int row_bytes, int rows) {
  const int rb = box_bytes(row_bytes);
  uint64_t dims[3] = {(uint64_t)rb, (uint64_t)rows, (uint64_t)(row_bytes / rb)};
  uint64_t strides[2] = {(uint64_t)row_bytes, (uint64_t)rb};
  uint32_t box[3] = {(uint32_t)rb, (uint32_t)kDecUnitRows, (uint32_t)(row_bytes / rb)};
  return encode_tiled(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, (void*)q, dims, strides, box,
                      rb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B) ==
         CUDA_SUCCESS;
}

static int num_sms() {
  static int cached[64] = {};
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev >= 0 && dev < 64 && cached[dev]) return cached[dev];
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    n = 148;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  // at most T*k <= 64 routed experts, each one tile (rows <= T <= BM), plus
  // the shared expert
  const int maxslots = 1 + (a.E < a.T * a.k ? a.E : a.T * a.k);
  if (a.T < 1 || a.T > kDecMaxRows || a.d % 128 || a.F % 128 || a.E > kMaxE || a.k > kMaxK ||
      a.BM < kDecMaxRows || maxslots > kMaxSlots)
    return cudaErrorInvalidValue;
  static bool attr_set = false;  // (idempotent: races only repeat the call)
  if (!attr_set) {
    carveout_max((const void*)dec_gateup_kernel);
    carveout_max((const void*)dec_down_kernel);
    attr_set = true;
  }
  CUtensorMap tg, tu, td;
  if (!codes_map(&tg, a.gq, a.d / 2, (a.E + 1) * a.F) ||
      !codes_map(&tu, a.uq, a.d / 2, (a.E + 1) * a.F) ||
      !codes_map(&td, a.dq, a.F / 2, (a.E + 1) * a.d))
    return cudaErrorInvalidValue;
  // gate/up: as many stages as fit beside the other regions
  int gst = kGuMaxStages;
  while (gst > 1 && gu_smem(a.T, a.E, a.d, gst).total > kGuSmemBudget) --gst;
  const size_t gsmem = gu_smem(a.T, a.E, a.d, gst).total;
  const int items = maxslots * (a.F / kDecUnitRows);
  const int ggrid = items < num_sms() ? items : num_sms();
  cudaError_t err = ensure_smem_attr((const void*)dec_gateup_kernel, gsmem);
  if (err != cudaSuccess) return err;
  prof_begin(K_DEC_GATEUP, s);
  err = launch_pdl(dec_gateup_kernel, dim3(ggrid), dim3(kDecThreads), gsmem, s, tg, tu, a, gst);
  prof_end(K_DEC_GATEUP, s);
  if (err != cudaSuccess) return err;
  // down: one stage per slot up to its budget
  int dst = (int)(kDnStageBudget / dn_stage_bytes(a.F));
  if (dst > maxslots) dst = maxslots;
  if (dst > kDnMaxStages) dst = kDnMaxStages;
  if (dst < 1) dst = 1;
  const size_t dsmem = dn_smem(a.T, a.E, a.F, dst).total;
  err = ensure_smem_attr((const void*)dec_down_kernel, dsmem);
  if (err != cudaSuccess) return err;
  prof_begin(K_DEC_DOWN, s);
  err = launch_pdl(dec_down_kernel, dim3(a.d / kDecUnitRows), dim3(kDecThreads), dsmem, s, td, a,
                   dst);
  prof_end(K_DEC_DOWN, s);
  return err;
}

}  // namespace lily
