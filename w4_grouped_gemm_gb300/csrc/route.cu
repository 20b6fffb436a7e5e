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
#include <algorithm>

#include "routing.cuh"

namespace lily {

// ============================================================== router logits
// logits[t][e] = sum_i x[t][i] * W[e][i] (+ b[e]), fp32 accumulation.

// ---------------------------------------------------------------- tensor cores
// logits = x * W^T with x (bf16, exact) and W = W_hi + W_mid + W_lo, three
// bf16 terms that together hold every bit of the fp32 W.  Each bf16 x bf16
// product is exact in fp32, so the tensor cores give fp32-accumulated logits
// of the fp32 weights.  Tokens are the M = 128 operand, experts the N operand;
// the K loop runs over (term, 64-wide block) pairs and is split across CTAs,
// each writing fp32 partial logits; a wide reduction kernel sums the splits
// in order (deterministic) and adds the bias.

__global__ void __launch_bounds__(256) router_prep_kernel(const float* __restrict__ w,
                                                          __nv_bfloat16* __restrict__ w3,
                                                          int64_t n_w) {
  pdl_wait();  // w3 may still be read by the predecessor (the previous layer's router)
  pdl_trigger();
  // four weights per thread: one 16-byte load, three 8-byte stores (n_w is a
  // multiple of 4: d is a multiple of 128; w is 16-byte aligned)
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_w / 4; i += stride) {
    const float4 v4 = reinterpret_cast<const float4*>(w)[i];
    const float v[4] = {v4.x, v4.y, v4.z, v4.w};
    __nv_bfloat16 hi[4], mid[4], lo[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      hi[u] = __float2bfloat16_rn(v[u]);
      const float r1 = v[u] - __bfloat162float(hi[u]);
      mid[u] = __float2bfloat16_rn(r1);
      lo[u] = __float2bfloat16_rn(r1 - __bfloat162float(mid[u]));
    }
    reinterpret_cast<uint2*>(w3)[i] = *reinterpret_cast<const uint2*>(hi);
    reinterpret_cast<uint2*>(w3 + n_w)[i] = *reinterpret_cast<const uint2*>(mid);
    reinterpret_cast<uint2*>(w3 + 2 * n_w)[i] = *reinterpret_cast<const uint2*>(lo);
  }
}

constexpr int kRtThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kRtStages = 4;
constexpr int kRtMaxSplits = 8;

int router_splits(int T, int d) {
  const int mt = (T + 127) / 128;
  const int ks = 3 * (d / 64);
  int S = (128 + mt - 1) / mt;
  if (S > kRtMaxSplits) S = kRtMaxSplits;
  if (S > ks / 2) S = ks / 2;
  return S < 1 ? 1 : S;
}

static int router_ne(int E) { return (E + 15) & ~15; }
// Experts per CTA: all of them, or -- while twice the CTAs still fit on the
// SMs at once, from 128 experts on in multiples of 32 -- half of them, two
// CTAs per token tile and split: twice the SMs pulling the split weights
// through, each half the bytes per step.  (With the grid already filling the
// SMs, a second wave measured slower: T = 2048 and 8192.)
static int router_nec(int E, int ctas, int sms) {
  const int NE = router_ne(E);
  return (NE >= 128 && NE % 32 == 0 && 2 * ctas <= sms) ? NE / 2 : NE;
}

static size_t router_tc_smem_nec(int NEc) {
  return 1024 + (size_t)kRtStages * (128 * 128 + NEc * 128) + 16 * 8 + 16;
}
size_t router_tc_smem(int E) { return router_tc_smem_nec(router_ne(E)); }

__global__ void __launch_bounds__(kRtThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                     int T, int d, int E, int NE, float* __restrict__ partial, uint32_t* status) {
  // NE: experts of this CTA (a multiple of 16), from expert n0 = blockIdx.z * NE
  extern __shared__ uint8_t smem_raw[];
  // aligned up to 1024 bytes by pointer arithmetic on the shared array, so
  // the compiler keeps the accesses in the shared window (not generic)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int ABYTES = 128 * 128, STAGE = ABYTES + NE * 128;
  uint64_t* full = (uint64_t*)(smem + kRtStages * STAGE);
  uint64_t* empty = full + kRtStages;
  uint64_t* accfull = empty + kRtStages;
  int* misc = (int*)(accfull + 1);
  volatile int* abort = misc;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * 128, split = blockIdx.y, S = gridDim.y, n0 = blockIdx.z * NE;
  const int KB = d / 64, KS = 3 * KB;
  const int ks0 = split * KS / S, nk = (split + 1) * KS / S - ks0;
  uint32_t tcols = 32;
  while ((int)tcols < NE) tcols <<= 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kRtStages; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    mbar_init(smem_u32(accfull), 1);
    misc[0] = 0;
    fence_mbar_init();
    prefetch_tensormap(&tm_x);
    prefetch_tensormap(&tm_w);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&misc[1]), tcols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = (uint32_t)misc[1];
  pdl_wait();  // the split weights and x come from before
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      int i = 0;
      for (; i < nk; ++i) {
        const int st = i % kRtStages;
        if (i >= kRtStages &&
            !mbar_wait(smem_u32(&empty[st]), ((i / kRtStages) + 1) & 1, abort, status))
          break;
        const int ks = ks0 + i, term = ks / KB, kb = ks % KB;
        const uint32_t fb = smem_u32(&full[st]);
        uint8_t* sp = smem + (size_t)st * STAGE;
        mbar_arrive_expect_tx(fb, (uint32_t)STAGE);
        tma_load_2d(smem_u32(sp), &tm_x, kb * 64, m0, fb);
        tma_load_2d(smem_u32(sp + ABYTES), &tm_w, kb * 64, term * E + n0, fb);
      }
      if (*abort) {  // let copies still in flight land before exit
        int never = 0;
        for (int k2 = (i > kRtStages ? i - kRtStages : 0); k2 < i; ++k2)
          mbar_wait(smem_u32(&full[k2 % kRtStages]), (k2 / kRtStages) & 1, &never, status);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // whole warp, warp-uniform operands; one elected lane issues the step
    const uint32_t idesc = idesc_bf16_f32(128, NE);
    for (int i = 0; i < nk; ++i) {
      const int st = i % kRtStages;
      if (!warp_wait_all(smem_u32(&full[st]), (i / kRtStages) & 1, abort, status)) break;
      tc_fence_after();
      const uint32_t a0 = smem_u32(smem + (size_t)st * STAGE);
      const uint64_t ad = sdesc_sw128(a0), bd = sdesc_sw128(a0 + ABYTES);
      if (elect_one()) {
#pragma unroll
        for (int k16 = 0; k16 < 4; ++k16)  // +32 B along K = +2 in each descriptor
          mma_f16(tmem, ad + 2 * k16, bd + 2 * k16, idesc, (i | k16) != 0);
        mma_commit(smem_u32(&empty[st]));
      }
      __syncwarp();
    }
    mma_commit_warp(smem_u32(accfull));
    __syncwarp();
  } else {
    int okv = 1;
    if (lane == 0) okv = mbar_wait(smem_u32(accfull), 0, abort, status) && !*abort;
    okv = __shfl_sync(0xffffffffu, okv, 0);
    if (okv) {
      tc_fence_after();
      const int q = warp & 3;
      const int t = m0 + q * 32 + lane;
      float* dst = partial + ((size_t)split * T + t) * E + n0;
      for (int cb = 0; cb < NE; cb += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + cb, v);
        tmem_ld_wait();
        if (t < T) {
          if ((E & 3) == 0 && cb + 32 <= NE && n0 + cb + 32 <= E) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4*>(dst + cb + j) =
                  make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                              __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (cb + j < NE && n0 + cb + j < E) dst[cb + j] = __uint_as_float(v[j]);
          }
        }
      }
    }
  }

  if (warp == 1 && lane == 0) {
    int never = 0;
    mbar_wait(smem_u32(accfull), 0, &never, status);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tcols);
  }
}

// logits[t][e] = sum_s partial[s][t][e] (+ b[e]), splits added in order;
// four logits per thread (E % 4 == 0) or one.
__global__ void __launch_bounds__(256) router_reduce_kernel(const float* __restrict__ partial,
                                                            int S, const float* __restrict__ b,
                                                            float* __restrict__ logits, int T,
                                                            int E) {
  pdl_wait();  // the partial logits come from the predecessor
  pdl_trigger();
  const int64_t n = (int64_t)T * E;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  if ((E & 3) == 0) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n / 4; i += stride) {
      // every split's load issued before the (in-order) sum
      float4 v[kRtMaxSplits];
#pragma unroll
      for (int sp = 0; sp < kRtMaxSplits; ++sp)
        if (sp < S) v[sp] = __ldcg(reinterpret_cast<const float4*>(partial + (int64_t)sp * n) + i);
      float4 acc = v[0];
#pragma unroll
      for (int sp = 1; sp < kRtMaxSplits; ++sp)
        if (sp < S) {
          acc.x += v[sp].x; acc.y += v[sp].y; acc.z += v[sp].z; acc.w += v[sp].w;
        }
      if (b) {
        const int e = (int)((4 * i) % E);
        acc.x += b[e]; acc.y += b[e + 1]; acc.z += b[e + 2]; acc.w += b[e + 3];
      }
      reinterpret_cast<float4*>(logits)[i] = acc;
    }
  } else {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += stride) {
      float acc = __ldcg(partial + i);
      for (int sp = 1; sp < S; ++sp) acc += __ldcg(partial + (int64_t)sp * n + i);
      if (b) acc += b[i % E];
      logits[i] = acc;
    }
  }
}

cudaError_t launch_router_split(const float* w, int E, int d, void* w_split, cudaStream_t s) {
  const int64_t n_w = (int64_t)E * d;
  int pblocks = (int)((n_w / 4 + 255) / 256);
  if (pblocks > 152 * 8) pblocks = 152 * 8;
  prof_begin(K_ROUTER_PREP, s);
  const cudaError_t err = launch_pdl(router_prep_kernel, dim3(pblocks), dim3(256), 0, s, w,
                                     static_cast<__nv_bfloat16*>(w_split), n_w);
  prof_end(K_ROUTER_PREP, s);
  return err;
}

cudaError_t launch_router_tc(const void* x, const float* w, const float* bias, int T, int d,
                             int E, void* w_split, const void* w_presplit, float* partial,
                             float* logits, uint32_t* status, cudaStream_t s) {
  // a split made once ahead (weights do not change between calls) replaces
  // the per-call split into the workspace
  void* wsp = w_presplit ? const_cast<void*>(w_presplit) : w_split;
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 0;
  const int ctas = ((T + 127) / 128) * router_splits(T, d);
  const int NEc = router_nec(E, ctas, sms), nN = router_ne(E) / NEc;
  CUtensorMap tm_x, tm_w;
  {
    uint64_t dims[2] = {(uint64_t)d, (uint64_t)T};
    uint64_t strides[1] = {(uint64_t)d * 2};
    uint32_t box[2] = {64, 128};
    if (encode_tiled(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (void*)x, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    uint64_t dims[2] = {(uint64_t)d, (uint64_t)3 * E};
    uint64_t strides[1] = {(uint64_t)d * 2};
    uint32_t box[2] = {64, (uint32_t)NEc};
    if (encode_tiled(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, wsp, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  cudaError_t err = cudaSuccess;
  if (!w_presplit) {
    err = launch_router_split(w, E, d, w_split, s);
    if (err != cudaSuccess) return err;
  }
  const size_t smem = router_tc_smem_nec(NEc);
  err = ensure_smem_attr((const void*)router_tc_kernel, smem);
  if (err != cudaSuccess) return err;
  dim3 grid((T + 127) / 128, router_splits(T, d), nN);
  prof_begin(K_ROUTER_GEMM, s);
  err = launch_pdl(router_tc_kernel, grid, dim3(kRtThreads), smem, s, tm_x, tm_w, T, d, E, NEc,
                   partial, status);
  prof_end(K_ROUTER_GEMM, s);
  if (err != cudaSuccess) return err;
  const int64_t nr = (E & 3) == 0 ? (int64_t)T * E / 4 : (int64_t)T * E;
  int rblocks = (int)((nr + 255) / 256);
  if (rblocks > 152 * 8) rblocks = 152 * 8;
  prof_begin(K_ROUTER_REDUCE, s);
  err = launch_pdl(router_reduce_kernel, dim3(rblocks), dim3(256), 0, s, partial, (int)grid.y,
                   bias, logits, T, E);
  prof_end(K_ROUTER_REDUCE, s);
  return err;
}

// ============================================================== routing kernel

// Grid-wide barrier for a cooperative launch (all blocks co-resident), with a
// bounded wait: a block that has waited limit_ns (2 s unless a test lowers
// it) gives up, flags LILY_STATUS_TIMEOUT and gets false, the same value in
// every thread of the block.  Its arrival is already counted, so the last
// block to arrive still resets the count and releases the generation; the
// barrier words end consistent for the next call either way.
__device__ bool grid_barrier(uint32_t* bar, uint32_t nblocks, uint32_t* status,
                             uint64_t limit_ns) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    volatile uint32_t* gen = bar + 1;
    uint32_t g = *gen;
    __threadfence();
    uint32_t arrived = atomicAdd(bar, 1u);
    if (arrived == nblocks - 1) {
      atomicExch(bar, 0u);
      __threadfence();
      atomicAdd(bar + 1, 1u);
    } else {
      const uint64_t t0 = globaltimer_ns();
      while (*gen == g) {
        if (globaltimer_ns() - t0 >= limit_ns) {
          set_status(status, LILY_STATUS_TIMEOUT);
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// Routing of tokens [blk * 8 * WT, ...) as block blk of nblk (the body of
// route_kernel; WT tokens per warp).  Needs kRouteThreads threads.
template <int WT>  // tokens per warp
__device__ __forceinline__ void route_body(const RouteArgs& a, int blk, int nblk) {
  constexpr int kBlkTok = 8 * WT;  // tokens per block
  static_assert(kBlkTok <= kRouteTok, "shared arrays hold kRouteTok tokens");
  __shared__ int s_ids[kRouteTok * kMaxK];
  __shared__ int s_rank[kRouteTok * kMaxK];
  __shared__ int s_cnt[kMaxE];
  __shared__ int s_before[kMaxE];
  __shared__ int s_off[kMaxE];
  __shared__ int s_scan_tmp[8];

  const int T = a.T, E = a.E, k = a.k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blk * kBlkTok;
  const int ntok = min(kBlkTok, T - t0);
  const int npair = ntok * k;

  // ---- phase 1: top-k + gates, one warp per token (4 tokens per warp)
  constexpr int kWarpTok = WT;
  // logits of this warp's tokens (lane holds experts lane + 32c), all loads
  // of the warp issued together
  float lv[kWarpTok][kMaxE / 32];
#pragma unroll
  for (int i = 0; i < kWarpTok; ++i) {
    const int tl = warp * kWarpTok + i;
#pragma unroll
    for (int c = 0; c < kMaxE / 32; ++c) {
      const int e = lane + 32 * c;
      lv[i][c] = (tl < ntok && e < E) ? __ldcg(a.logits_src + (size_t)(t0 + tl) * E + e) : 0.f;
    }
  }
  if (a.logits_dst != a.logits_src) {
#pragma unroll
    for (int i = 0; i < kWarpTok; ++i) {
      const int tl = warp * kWarpTok + i;
#pragma unroll
      for (int c = 0; c < kMaxE / 32; ++c)
        if (tl < ntok && lane + 32 * c < E) a.logits_dst[(size_t)(t0 + tl) * E + lane + 32 * c] = lv[i][c];
    }
  }
  // the warp's tokens' selections interleaved (tokens past the end select
  // from zeros and are not stored)
  int my_id[kWarpTok];
  float my_gate[kWarpTok];
  const uint32_t nan_mask = warp_topk_multi<kWarpTok>(lv, E, k, my_id, my_gate);
#pragma unroll
  for (int i = 0; i < kWarpTok; ++i) {
    const int tl = warp * kWarpTok + i;
    if (tl >= ntok) break;
    const int t = t0 + tl;
    if (((nan_mask >> i) & 1u) && lane == 0) set_status(a.status, LILY_STATUS_NAN_LOGIT);
    if (lane < k) {
      a.ids[(size_t)t * k + lane] = my_id[i];
      a.gates[(size_t)t * k + lane] = my_gate[i];
      s_ids[tl * k + lane] = my_id[i];
    }
  }
  // ---- phase 2: block histogram and stable local rank of each pair (one
  // pair per thread): the rank among the warp's pairs of the same expert
  // from a match, plus that expert's pairs in the earlier warps
  static_assert(kRouteTok * kMaxK <= kRouteThreads, "one pair per thread");
  constexpr int kRouteWarps = kRouteThreads / 32;
  __shared__ int s_wcnt[kRouteWarps][kMaxE];
  for (int i = threadIdx.x; i < kRouteWarps * kMaxE; i += kRouteThreads) (&s_wcnt[0][0])[i] = 0;
  __syncthreads();
  {
    const int q = threadIdx.x;
    const int e = q < npair ? s_ids[q] : -1;
    const unsigned same = __match_any_sync(0xffffffffu, e);
    const int lrank = __popc(same & ((1u << lane) - 1u));
    if (e >= 0 && lrank == 0) s_wcnt[warp][e] = __popc(same);
    __syncthreads();
    if (e >= 0) {
      int rk = lrank;
      for (int w2 = 0; w2 < warp; ++w2) rk += s_wcnt[w2][e];
      s_rank[q] = rk;
    }
    for (int e2 = threadIdx.x; e2 < E; e2 += kRouteThreads) {
      int c = 0;
#pragma unroll
      for (int w2 = 0; w2 < kRouteWarps; ++w2) c += s_wcnt[w2][e2];
      s_cnt[e2] = c;
    }
  }
  __syncthreads();
  if (nblk > 1) {
    for (int e = threadIdx.x; e < E; e += kRouteThreads) a.hist[(size_t)blk * E + e] = s_cnt[e];

    // a block whose wait ran out leaves every output of its pairs unwritten:
    // the other blocks' histogram rows may not have been written yet
    if (!grid_barrier(a.bar, nblk, a.status, a.wait_ns)) return;

    // ---- phase 3: global counts, scan, this block's bases, scatter
    for (int e = threadIdx.x; e < kMaxE; e += kRouteThreads) {
      int cnt = 0, before = 0;
      if (e < E) {
#pragma unroll 16
        for (int b = 0; b < nblk; ++b) {
          int h = __ldcg(&a.hist[(size_t)b * E + e]);
          cnt += h;
          before += (b < blk) ? h : 0;
        }
      }
      s_cnt[e] = cnt;
      s_before[e] = before;
    }
  } else {  // one block: its histogram is the global one
    for (int e = threadIdx.x; e < kMaxE; e += kRouteThreads) {
      if (e >= E) s_cnt[e] = 0;
      s_before[e] = 0;
    }
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

template <int WT>
__global__ void __launch_bounds__(kRouteThreads, 4) route_kernel(RouteArgs a) {
  pdl_wait();  // the logits come from the predecessor
  pdl_trigger();
  route_body<WT>(a, blockIdx.x, gridDim.x);
}

int route_max_blocks() {
  static int cached[64] = {};
  int dev = 0, nsm = 0, per = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64 && cached[dev]) return cached[dev];
  if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, route_kernel<4>, kRouteThreads, 0) !=
      cudaSuccess)
    return 0;
  if (dev >= 0 && dev < 64) cached[dev] = nsm * per;
  return nsm * per;
}

template <int WT>
static cudaError_t launch_route_wt(const RouteArgs& a, cudaStream_t s) {
  const int nblk = (a.T + 8 * WT - 1) / (8 * WT);
  RouteArgs args = a;
  void* params[] = {&args};
  // one block needs no co-residency guarantee: a plain launch is cheaper
  return nblk == 1 ? launch_pdl(route_kernel<WT>, dim3(1), dim3(kRouteThreads), 0, s, args)
                   : cudaLaunchCooperativeKernel((const void*)route_kernel<WT>, dim3(nblk),
                                                 dim3(kRouteThreads), params, 0, s);
}

cudaError_t launch_route(const RouteArgs& a, cudaStream_t s) {
  prof_begin(K_ROUTE, s);
  const cudaError_t err =
      route_tok(a.T) == 16 ? launch_route_wt<2>(a, s) : launch_route_wt<4>(a, s);
  prof_end(K_ROUTE, s);
  return err;
}

}  // namespace lily
