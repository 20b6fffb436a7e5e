// decode.cu -- W4 GEMV path for batch-1 / small-batch decode (1..8 rows).
//
// Batch-1 decode is bandwidth-bound, so the aim is the fewest bytes and the
// fewest instructions per weight byte (page "Lily Beats MLX-LM 1.35x on
// Decode: Perplexity's Rust+Metal Engine for Apple Silicon", section "Decode:
// eliminating per-token CPU round trips"; verify batches of two to five rows
// are the speculative-decoding shapes of the same section).  Each distinct
// active expert (block-map tile) is streamed once for all its rows.
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
// laid out in that same order (x staged in shared memory; H written in it by
// the gate/up kernel), so the K order of both operands agrees.
#include "common.cuh"

namespace lily {

constexpr int kDecThreads = 256;
constexpr int kDecMaxRows = 8;  // mma N

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

// Which tile a decode CTA serves: the routing's plan entry of the slot
// (slot 0 = shared expert, slot i >= 1 = block-map tile i-1), one 16-byte
// load.  Returns false if the slot is unused.
__device__ __forceinline__ bool decode_tile(const DecodeArgs& a, int slot, int& expert, int& row0,
                                            int& rows) {
  const int4 h = __ldcg(reinterpret_cast<const int4*>(a.plan + (size_t)slot * kPlanWords));
  expert = h.x;
  row0 = h.y;
  rows = h.z;
  if (rows <= 0) return false;
  if (expert < 0 || expert > a.E || rows > kDecMaxRows) {
    if (threadIdx.x == 0) set_status(a.status, LILY_STATUS_BAD_TILE);
    return false;
  }
  return true;
}
// Token and gate of row n of a slot (from the plan).
__device__ __forceinline__ int plan_token(const DecodeArgs& a, int slot, int n) {
  return __ldcg(a.plan + (size_t)slot * kPlanWords + 8 + n);
}
__device__ __forceinline__ float plan_gate(const DecodeArgs& a, int slot, int n) {
  return __int_as_float(__ldcg(a.plan + (size_t)slot * kPlanWords + 16 + n));
}

// Up to kChunk groups of 16 weight rows [r0, r0+16) of one packed matrix
// (row length K): the codes of rows gi and gi+8 for this lane's 8 K values,
// and the rows' scales and biases, loaded into registers ahead of use so the
// loads of a chunk are in flight together.
constexpr int kChunk = 4;
struct WChunk {
  uint2 wa[kChunk], wb[kChunk];
  float sa[kChunk], sb[kChunk], ba[kChunk], bb[kChunk];
};
__device__ __forceinline__ void load_wchunk(WChunk& w, const uint8_t* __restrict__ q,
                                            const uint16_t* __restrict__ s,
                                            const uint16_t* __restrict__ b, size_t r0, int K,
                                            int g0, int gstep) {
  const int lane = threadIdx.x & 31, gi = lane >> 2, c = lane & 3;
  const int G = K / 64;
  const uint8_t* qa = q + (r0 + gi) * (size_t)(K / 2) + c * 8;
  const uint8_t* qb = qa + 8 * (size_t)(K / 2);
  const uint16_t* sa = s + (r0 + gi) * (size_t)G;
  const uint16_t* ba = b + (r0 + gi) * (size_t)G;
#pragma unroll
  for (int i = 0; i < kChunk; ++i) {
    const int g = g0 + i * gstep;
    if (g < G) {
      w.wa[i] = __ldcs(reinterpret_cast<const uint2*>(qa + g * 32));
      w.wb[i] = __ldcs(reinterpret_cast<const uint2*>(qb + g * 32));
      w.sa[i] = bf16_bits_to_float(__ldg(sa + g));
      w.sb[i] = bf16_bits_to_float(__ldg(sa + 8 * G + g));
      w.ba[i] = bf16_bits_to_float(__ldg(ba + g));
      w.bb[i] = bf16_bits_to_float(__ldg(ba + 8 * G + g));
    }
  }
}
// Group i of a loaded chunk against B fragments xw (8 words: this lane's
// (i, i+4) pairs) and the group sums x0, x1 of accumulator columns 2c, 2c+1.
template <bool F16>
__device__ __forceinline__ void chunk_group(const WChunk& w, int i, const uint32_t (&xw)[8],
                                            float x0, float x1, float (&out)[4]) {
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t pa[4], pb[4];
    code_pairs<F16>(h == 0 ? w.wa[i].x : w.wa[i].y, pa);
    code_pairs<F16>(h == 0 ? w.wb[i].x : w.wb[i].y, pb);
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const uint32_t afrag[4] = {pa[2 * m], pb[2 * m], pa[2 * m + 1], pb[2 * m + 1]};
      mma_16816<F16>(acc, afrag, xw[h * 4 + m * 2], xw[h * 4 + m * 2 + 1]);
    }
  }
  constexpr float off = F16 ? 1024.f : 128.f;  // the code offset of the magic
  out[0] += w.sa[i] * (acc[0] - off * x0) + w.ba[i] * x0;
  out[1] += w.sa[i] * (acc[1] - off * x1) + w.ba[i] * x1;
  out[2] += w.sb[i] * (acc[2] - off * x0) + w.bb[i] * x0;
  out[3] += w.sb[i] * (acc[3] - off * x1) + w.bb[i] * x1;
}

// Gate/up: CTA = (tile slot, 16 features); 8 warps split K; H = silu(g) * u.
// B fragments and group sums come from x in fragment order (xpg, xsg, written
// by the router launch), so no activation staging is needed.
__global__ void __launch_bounds__(kDecThreads) dec_gateup_kernel(const DecodeArgs a) {
  __shared__ float part[8][2][16][kDecMaxRows];  // per-warp partial outputs
  __shared__ int tok[kDecMaxRows];
  const int G = a.d / 64;
  const int nfb = a.F / 16;
  const int slot = blockIdx.x / nfb, fb = blockIdx.x % nfb;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gi = lane >> 2, c = lane & 3;
  // this warp's first chunk of weight groups (g = warp, warp + 8, ...); the
  // shared expert's (slot 0) goes before the wait for the routing
  WChunk wg, wu;
  if (slot == 0) {
    const size_t r0s = (size_t)a.E * a.F + (size_t)fb * 16;
    load_wchunk(wg, a.gq, a.gs, a.gb, r0s, a.d, warp, 8);
    load_wchunk(wu, a.uq, a.us, a.ub, r0s, a.d, warp, 8);
  }
  pdl_wait();
  pdl_trigger();
  int expert, row0, rows;
  if (!decode_tile(a, slot, expert, row0, rows)) return;
  const size_t r0 = (size_t)expert * a.F + (size_t)fb * 16;
  if (slot != 0) {
    load_wchunk(wg, a.gq, a.gs, a.gb, r0, a.d, warp, 8);
    load_wchunk(wu, a.uq, a.us, a.ub, r0, a.d, warp, 8);
  }
  if (threadIdx.x < kDecMaxRows) tok[threadIdx.x] = plan_token(a, slot, min((int)threadIdx.x, rows - 1));
  __syncthreads();
  // B-fragment row of this lane: slot row gi (zero beyond the slot's rows);
  // group sums of accumulator columns 2c, 2c+1
  const uint32_t* xrow = a.xpg + (size_t)tok[min(gi, rows - 1)] * G * 32 + c * 8;
  const float* xs0 = a.xsg + (size_t)tok[min(2 * c, rows - 1)] * G;
  const float* xs1 = a.xsg + (size_t)tok[min(2 * c + 1, rows - 1)] * G;
  float og[4] = {0.f, 0.f, 0.f, 0.f}, ou[4] = {0.f, 0.f, 0.f, 0.f};
  for (int g0 = warp; g0 < G; g0 += 8 * kChunk) {
    if (g0 != warp) {
      load_wchunk(wg, a.gq, a.gs, a.gb, r0, a.d, g0, 8);
      load_wchunk(wu, a.uq, a.us, a.ub, r0, a.d, g0, 8);
    }
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      const int g = g0 + 8 * i;
      if (g < G) {
        uint4 h0 = make_uint4(0, 0, 0, 0), h1 = h0;
        if (gi < rows) {
          h0 = __ldg(reinterpret_cast<const uint4*>(xrow + (size_t)g * 32));
          h1 = __ldg(reinterpret_cast<const uint4*>(xrow + (size_t)g * 32 + 4));
        }
        const uint32_t xw[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
        const float x0 = 2 * c < rows ? __ldg(xs0 + g) : 0.f;
        const float x1 = 2 * c + 1 < rows ? __ldg(xs1 + g) : 0.f;
        chunk_group<false>(wg, i, xw, x0, x1, og);
        chunk_group<false>(wu, i, xw, x0, x1, ou);
      }
    }
  }
  part[warp][0][gi][2 * c] = og[0];
  part[warp][0][gi][2 * c + 1] = og[1];
  part[warp][0][gi + 8][2 * c] = og[2];
  part[warp][0][gi + 8][2 * c + 1] = og[3];
  part[warp][1][gi][2 * c] = ou[0];
  part[warp][1][gi][2 * c + 1] = ou[1];
  part[warp][1][gi + 8][2 * c] = ou[2];
  part[warp][1][gi + 8][2 * c + 1] = ou[3];
  __syncthreads();
  if (threadIdx.x < 16 * kDecMaxRows) {
    const int row = threadIdx.x / kDecMaxRows, n = threadIdx.x % kDecMaxRows;
    float g = 0.f, u = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      g += part[w][0][row][n];
      u += part[w][1][row][n];
    }
    if (n < rows) {
      const float h = g / (1.f + __expf(-g)) * u;
      if (!(fabsf(h) <= 65504.f)) set_status(a.status, LILY_STATUS_F16_RANGE);
      const int f = fb * 16 + row;  // H row in pair order, one 64-group after another
      static_cast<__half*>(a.H)[(size_t)(row0 + n) * a.F + (f & ~63) + hpair_pos(f & 63)] =
          __float2half_rn(h);
    }
  }
}

// Down + combine: CTA = 16 output features over every active tile slot; warp
// w of 16 takes slots w, w + 16, ...  For each slot it runs the 16-row W4
// GEMV over K = F against that slot's H rows (B fragments loaded straight
// from H, kept in pair order by the gate/up kernel; group sums X_g from the
// same loads), with the next chunk of weight groups in flight, then adds
// gate * out into its own [token][feature] tile in shared memory.  The tiles
// are summed in warp order, so the result is deterministic.
constexpr int kDownWarps = 16;
__global__ void __launch_bounds__(32 * kDownWarps) dec_down_combine_kernel(const DecodeArgs a) {
  __shared__ float ytile[kDownWarps][kDecMaxRows][16];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gi = lane >> 2, c = lane & 3;
  const int G = a.F / 64;
  const int f0 = blockIdx.x * 16;  // output features [f0, f0 + 16)
  pdl_wait();
  pdl_trigger();
  for (int i = threadIdx.x; i < kDownWarps * kDecMaxRows * 16; i += blockDim.x)
    (&ytile[0][0][0])[i] = 0.f;
  __syncthreads();
  const int nslots = 1 + a.cap;  // unused slots have rows = 0 in the plan
  const uint16_t* H = static_cast<const uint16_t*>(a.H);
  for (int slot = warp; slot < nslots; slot += kDownWarps) {
    int expert, row0, rows;
    if (!decode_tile(a, slot, expert, row0, rows)) continue;
    const size_t r0 = (size_t)expert * a.d + f0;
    // this lane's B-fragment row: slot row n = gi (zero beyond the slot's rows)
    const uint16_t* hrow = H + (size_t)(row0 + min(gi, rows - 1)) * a.F + c * 16;
    WChunk wd, wn;
    load_wchunk(wd, a.dq, a.ds, a.db, r0, a.F, 0, 1);
    float o[4] = {0.f, 0.f, 0.f, 0.f};
    for (int g0 = 0; g0 < G; g0 += kChunk) {
      uint4 hh[kChunk][2];
#pragma unroll
      for (int i = 0; i < kChunk; ++i) {
        hh[i][0] = hh[i][1] = make_uint4(0, 0, 0, 0);
        if (g0 + i < G && gi < rows) {
          hh[i][0] = *reinterpret_cast<const uint4*>(hrow + (g0 + i) * 64);
          hh[i][1] = *reinterpret_cast<const uint4*>(hrow + (g0 + i) * 64 + 8);
        }
      }
      if (g0 + kChunk < G) load_wchunk(wn, a.dq, a.ds, a.db, r0, a.F, g0 + kChunk, 1);
#pragma unroll
      for (int i = 0; i < kChunk; ++i) {
        if (g0 + i < G) {
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
          chunk_group<true>(wd, i, xw, x0, x1, o);
        }
      }
      wd = wn;
    }
    // gate * out into this warp's tile: slot row n -> its token and gate
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int n = 2 * c + h;
      if (n < rows) {
        const int tok = plan_token(a, slot, n);
        const float gate = plan_gate(a, slot, n);
        ytile[warp][tok][gi] += gate * o[h];
        ytile[warp][tok][gi + 8] += gate * o[2 + h];
      }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < a.T * 16; i += blockDim.x) {
    const int t = i >> 4, f = i & 15;
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < kDownWarps; ++w) acc += ytile[w][t][f];
    if (a.y_f32)
      static_cast<float*>(a.y)[(size_t)t * a.d + f0 + f] = acc;
    else
      static_cast<__nv_bfloat16*>(a.y)[(size_t)t * a.d + f0 + f] = __float2bfloat16_rn(acc);
  }
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  if (a.T < 1 || a.T > kDecMaxRows || a.d % 16) return cudaErrorInvalidValue;
  const int slots = 1 + a.cap;
  prof_begin(K_DEC_GATEUP, s);
  cudaError_t err =
      launch_pdl(dec_gateup_kernel, dim3(slots * (a.F / 16)), dim3(kDecThreads), 0, s, a);
  prof_end(K_DEC_GATEUP, s);
  if (err != cudaSuccess) return err;
  prof_begin(K_DEC_DOWN, s);
  err = launch_pdl(dec_down_combine_kernel, dim3(a.d / 16), dim3(32 * kDownWarps), 0, s, a);
  prof_end(K_DEC_DOWN, s);
  return err;
}

}  // namespace lily
