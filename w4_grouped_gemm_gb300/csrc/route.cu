// route.cu -- GPU-resident MoE routing for sm_103a.
//
// Router logits, then one cooperative kernel that does top-k selection with
// renormalised softmax gates, the per-expert histogram, the exclusive prefix
// scan, the stable scatter of (token, slot) pairs into expert-contiguous rows
// and the tile block map -- all on the launch stream, with no host sync
// (page "Lily Beats MLX-LM 1.35x on Decode: Perplexity's Rust+Metal Engine for
// Apple Silicon", section "Prefill: fusing dequantisation and keeping routing
// GPU-resident": histogram, prefix scan, scatter and block map stay on the GPU;
// section "Model structure and three workload shapes": a router scores 256
// experts and picks eight).
#include "common.cuh"

namespace lily {

// ============================================================== router logits
// logits[t][e] = sum_i x[t][i] * W[e][i] (+ b[e]), fp32 accumulation.
// Both kernels also write x16, the fp16 copy of x that the grouped GEMM's
// tensor-core operand uses (exact for |x| in [2^-17, 65504]; larger values
// set LILY_STATUS_F16_RANGE).

__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t v, bool& ok) {
  const float lo = __uint_as_float(v << 16), hi = __uint_as_float(v & 0xFFFF0000u);
  ok &= fabsf(lo) <= 65504.f && fabsf(hi) <= 65504.f;
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Small T (decode): one warp per expert row, all tokens at once.
constexpr int kGemvMaxT = 8;
__global__ void __launch_bounds__(256) router_gemv_kernel(const __nv_bfloat16* __restrict__ x,
                                                          const float* __restrict__ w,
                                                          const float* __restrict__ b,
                                                          float* __restrict__ logits, int T,
                                                          int d, int E, uint32_t* __restrict__ x16,
                                                          uint32_t* status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (blockIdx.x == 0 && x16) {  // fp16 copy of the (few) rows
    bool ok = true;
    const uint32_t* xs = reinterpret_cast<const uint32_t*>(x);
    for (int i = threadIdx.x; i < T * d / 2; i += blockDim.x) x16[i] = bf2_to_h2(xs[i], ok);
    if (!ok) set_status(status, LILY_STATUS_F16_RANGE);
  }
  const int e = blockIdx.x * 8 + warp;
  if (e >= E) return;
  float acc[kGemvMaxT];
#pragma unroll
  for (int t = 0; t < kGemvMaxT; ++t) acc[t] = 0.f;
  const float4* wr = reinterpret_cast<const float4*>(w + (size_t)e * d);
  for (int i4 = lane; i4 < d / 4; i4 += 32) {
    float4 wv = __ldg(wr + i4);
#pragma unroll
    for (int t = 0; t < kGemvMaxT; ++t) {
      if (t < T) {
        const __nv_bfloat162* xp =
            reinterpret_cast<const __nv_bfloat162*>(x + (size_t)t * d + 4 * i4);
        float2 x01 = __bfloat1622float2(xp[0]);
        float2 x23 = __bfloat1622float2(xp[1]);
        acc[t] = fmaf(wv.x, x01.x, acc[t]);
        acc[t] = fmaf(wv.y, x01.y, acc[t]);
        acc[t] = fmaf(wv.z, x23.x, acc[t]);
        acc[t] = fmaf(wv.w, x23.y, acc[t]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kGemvMaxT; ++t) {
    float v = acc[t];
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0 && t < T) logits[(size_t)t * E + e] = v + (b ? b[e] : 0.f);
  }
}

// Larger T: 64 tokens x 64 experts per block, 4x4 outputs per thread.
constexpr int RG_BT = 64, RG_BE = 64, RG_BK = 32;
__global__ void __launch_bounds__(256) router_gemm_kernel(const __nv_bfloat16* __restrict__ x,
                                                          const float* __restrict__ w,
                                                          const float* __restrict__ b,
                                                          float* __restrict__ logits, int T,
                                                          int d, int E, uint32_t* __restrict__ x16,
                                                          uint32_t* status) {
  bool range_ok = true;
  __shared__ float xs[RG_BK][RG_BT + 4];
  __shared__ float ws[RG_BK][RG_BE + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int t0 = blockIdx.x * RG_BT, e0 = blockIdx.y * RG_BE;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < d; k0 += RG_BK) {
    {  // x tile: 64 tokens x 32 k, 8 bf16 per thread
      int row = threadIdx.x >> 2, kc = (threadIdx.x & 3) * 8;
      int t = t0 + row;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (t < T) v = *reinterpret_cast<const uint4*>(x + (size_t)t * d + k0 + kc);
      if (t < T && blockIdx.y == 0 && x16) {
        uint4 hv;
        hv.x = bf2_to_h2(v.x, range_ok);
        hv.y = bf2_to_h2(v.y, range_ok);
        hv.z = bf2_to_h2(v.z, range_ok);
        hv.w = bf2_to_h2(v.w, range_ok);
        *reinterpret_cast<uint4*>(x16 + ((size_t)t * d + k0 + kc) / 2) = hv;
      }
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float2 f = __bfloat1622float2(h[j]);
        xs[kc + 2 * j][row] = f.x;
        xs[kc + 2 * j + 1][row] = f.y;
      }
    }
    {  // w tile: 64 experts x 32 k, 8 floats per thread
      int row = threadIdx.x >> 2, kc = (threadIdx.x & 3) * 8;
      int e = e0 + row;
      float4 v0 = make_float4(0, 0, 0, 0), v1 = v0;
      if (e < E) {
        const float4* p = reinterpret_cast<const float4*>(w + (size_t)e * d + k0 + kc);
        v0 = __ldg(p);
        v1 = __ldg(p + 1);
      }
      ws[kc + 0][row] = v0.x; ws[kc + 1][row] = v0.y; ws[kc + 2][row] = v0.z; ws[kc + 3][row] = v0.w;
      ws[kc + 4][row] = v1.x; ws[kc + 5][row] = v1.y; ws[kc + 6][row] = v1.z; ws[kc + 7][row] = v1.w;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < RG_BK; ++kk) {
      float a[4], c[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = xs[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) c[j] = ws[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], c[j], acc[i][j]);
    }
    __syncthreads();
  }
  if (!range_ok) set_status(status, LILY_STATUS_F16_RANGE);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int e = e0 + tx * 4 + j;
      if (e < E) logits[(size_t)t * E + e] = acc[i][j] + (b ? b[e] : 0.f);
    }
  }
}

cudaError_t launch_router_logits(const void* x, const float* w, const float* b, float* logits,
                                 int T, int d, int E, void* x16, uint32_t* status,
                                 cudaStream_t s) {
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  uint32_t* x16w = static_cast<uint32_t*>(x16);
  if (T <= kGemvMaxT) {
    prof_begin(K_ROUTER_GEMV, s);
    router_gemv_kernel<<<(E + 7) / 8, 256, 0, s>>>(xb, w, b, logits, T, d, E, x16w, status);
    prof_end(K_ROUTER_GEMV, s);
  } else {
    prof_begin(K_ROUTER_GEMM, s);
    dim3 grid((T + RG_BT - 1) / RG_BT, (E + RG_BE - 1) / RG_BE);
    router_gemm_kernel<<<grid, 256, 0, s>>>(xb, w, b, logits, T, d, E, x16w, status);
    prof_end(K_ROUTER_GEMM, s);
  }
  return cudaGetLastError();
}

// ============================================================== routing kernel

// Order-preserving key of a logit: larger key = ranks first.  -0 and +0 map
// to the same key; a NaN maps to 0, below every number.
__device__ __forceinline__ uint32_t logit_key(float v) {
  if (v != v) return 0u;
  uint32_t u = __float_as_uint(v == 0.f ? 0.f : v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}

// Exclusive scan of one int per thread over a 256-thread block.
__device__ int block_exclusive_scan(int v, int* tmp /* [8] */) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) tmp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < kRouteThreads / 32) ? tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      int n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    if (lane < kRouteThreads / 32) tmp[lane] = w;  // inclusive warp totals
  }
  __syncthreads();
  int base = (warp > 0) ? tmp[warp - 1] : 0;
  int out = base + incl - v;
  __syncthreads();
  return out;
}

// Grid-wide barrier for a cooperative launch (all blocks co-resident), with a
// bounded wait: gives up after ~2 s and flags LILY_STATUS_TIMEOUT.
__device__ void grid_barrier(uint32_t* bar, uint32_t nblocks, uint32_t* status) {
  __syncthreads();
  if (threadIdx.x == 0) {
    volatile uint32_t* gen = bar + 1;
    uint32_t g = *gen;
    __threadfence();
    uint32_t arrived = atomicAdd(bar, 1u);
    if (arrived == nblocks - 1) {
      atomicExch(bar, 0u);
      __threadfence();
      atomicAdd(bar + 1, 1u);
    } else {
      uint64_t t0 = globaltimer_ns();
      while (*gen == g) {
        __nanosleep(64);
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          set_status(status, LILY_STATUS_TIMEOUT);
          break;
        }
      }
    }
    __threadfence();
  }
  __syncthreads();
}

constexpr int kMaxE = 256, kMaxK = 8;

__global__ void __launch_bounds__(kRouteThreads) route_kernel(RouteArgs a) {
  __shared__ int s_ids[kRouteTok * kMaxK];
  __shared__ int s_rank[kRouteTok * kMaxK];
  __shared__ int s_cnt[kMaxE];
  __shared__ int s_before[kMaxE];
  __shared__ int s_off[kMaxE];
  __shared__ int s_scan_tmp[8];

  const int T = a.T, E = a.E, k = a.k;
  const int blk = blockIdx.x, nblk = gridDim.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blk * kRouteTok;
  const int ntok = min(kRouteTok, T - t0);
  const int npair = ntok * k;

  // ---- phase 1: top-k + gates, one warp per token (4 tokens per warp)
  for (int i = 0; i < kRouteTok / 8; ++i) {
    const int tl = warp * (kRouteTok / 8) + i;
    if (tl >= ntok) break;
    const int t = t0 + tl;
    uint32_t key[kMaxE / 32];
    uint32_t avail = 0;
    bool saw_nan = false;
#pragma unroll
    for (int c = 0; c < kMaxE / 32; ++c) {
      const int e = lane + 32 * c;
      key[c] = 0;
      if (e < E) {
        float v = a.logits_src[(size_t)t * E + e];
        if (a.logits_dst != a.logits_src) a.logits_dst[(size_t)t * E + e] = v;
        saw_nan |= (v != v);
        key[c] = logit_key(v);
        avail |= 1u << c;
      }
    }
    if (__any_sync(0xffffffffu, saw_nan) && lane == 0) set_status(a.status, LILY_STATUS_NAN_LOGIT);
    float my_logit = 0.f;
    int my_id = 0;
    for (int j = 0; j < k; ++j) {
      // lane-local best: largest key, lowest id on ties (c ascending = id ascending)
      uint32_t bk = 0;
      int bc = -1;
#pragma unroll
      for (int c = 0; c < kMaxE / 32; ++c)
        if ((avail >> c) & 1u)
          if (bc < 0 || key[c] > bk) { bk = key[c]; bc = c; }
      const uint32_t kmax = __reduce_max_sync(0xffffffffu, bc >= 0 ? bk : 0u);
      const uint32_t cand = (bc >= 0 && bk == kmax) ? (uint32_t)(lane + 32 * bc) : 0xFFFFFFFFu;
      const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
      if ((int)(win & 31u) == lane) avail &= ~(1u << (win >> 5));
      if (lane == j) { my_logit = key_logit(kmax); my_id = (int)win; }
    }
    // gates: softmax over the kept logits; entries equal to the largest weigh 1
    const float lmax = __shfl_sync(0xffffffffu, my_logit, 0);
    float wgt = 0.f;
    if (lane < k) wgt = (my_logit == lmax) ? 1.f : expf(my_logit - lmax);
    float z = wgt;
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    if (lane < k) {
      a.ids[(size_t)t * k + lane] = my_id;
      a.gates[(size_t)t * k + lane] = wgt / z;
      s_ids[tl * k + lane] = my_id;
    }
  }
  for (int e = threadIdx.x; e < E; e += kRouteThreads) s_cnt[e] = 0;
  __syncthreads();

  // ---- phase 2: block histogram and stable local rank of each pair
  for (int q = threadIdx.x; q < npair; q += kRouteThreads) {
    const int e = s_ids[q];
    int r = 0;
    for (int q2 = 0; q2 < q; ++q2) r += (s_ids[q2] == e);
    s_rank[q] = r;
    atomicAdd(&s_cnt[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kRouteThreads) a.hist[(size_t)blk * E + e] = s_cnt[e];

  grid_barrier(a.bar, nblk, a.status);

  // ---- phase 3: global counts, scan, this block's bases, scatter
  for (int e = threadIdx.x; e < kMaxE; e += kRouteThreads) {
    int cnt = 0, before = 0;
    if (e < E) {
      for (int b = 0; b < nblk; ++b) {
        int h = __ldcg(&a.hist[(size_t)b * E + e]);
        cnt += h;
        before += (b < blk) ? h : 0;
      }
    }
    s_cnt[e] = cnt;
    s_before[e] = before;
  }
  __syncthreads();
  // kRouteThreads == kMaxE: one expert per thread
  const int e_me = threadIdx.x;
  const int off_me = block_exclusive_scan(s_cnt[e_me], s_scan_tmp);
  s_off[e_me] = off_me;
  __syncthreads();
  for (int q = threadIdx.x; q < npair; q += kRouteThreads) {
    const int e = s_ids[q];
    const int pos = s_off[e] + s_before[e] + s_rank[q];
    const int p = t0 * k + q;
    a.perm[pos] = p;
    a.inv[p] = pos;
  }

  // ---- block 0: counts, offsets and the block map
  if (blk == 0) {
    const int cnt = s_cnt[e_me];
    if (e_me < E) {
      a.counts[e_me] = cnt;
      a.offsets[e_me] = off_me;
    }
    if (e_me == 0) a.offsets[E] = T * k;
    const int ntile = (e_me < E) ? (cnt + a.BM - 1) / a.BM : 0;
    const int toff = block_exclusive_scan(ntile, s_scan_tmp);
    for (int i = 0; i < ntile; ++i) {
      a.block_map[2 * (toff + i)] = e_me;
      a.block_map[2 * (toff + i) + 1] = off_me + i * a.BM;
    }
    if (e_me == kMaxE - 1) *a.n_tiles = toff + ntile;
    const int total = __shfl_sync(0xffffffffu, toff + ntile, 31);  // valid in the last warp
    __shared__ int s_total;
    if (e_me == kMaxE - 1) s_total = total;
    __syncthreads();
    for (int i = s_total + threadIdx.x; i < a.cap; i += kRouteThreads) {
      a.block_map[2 * i] = -1;
      a.block_map[2 * i + 1] = -1;
    }
  }
}

int route_max_blocks() {
  int dev = 0, nsm = 0, per = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, route_kernel, kRouteThreads, 0) !=
      cudaSuccess)
    return 0;
  return nsm * per;
}

cudaError_t launch_route(const RouteArgs& a, cudaStream_t s) {
  const int nblk = (a.T + kRouteTok - 1) / kRouteTok;
  RouteArgs args = a;
  void* params[] = {&args};
  prof_begin(K_ROUTE, s);
  cudaError_t err = cudaLaunchCooperativeKernel((const void*)route_kernel, dim3(nblk),
                                                dim3(kRouteThreads), params, 0, s);
  prof_end(K_ROUTE, s);
  return err;
}

}  // namespace lily
