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
// laid out in shared memory in that same order, so the K order of both
// operands agrees.
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
template <bool F16>
__device__ __forceinline__ float act_to_float(uint16_t h) {
  return F16 ? __half2float(__ushort_as_half(h)) : bf16_bits_to_float(h);
}

// Which tile a decode CTA serves.  Slot 0 = shared expert (rows P..P+T-1);
// slot i >= 1 = block-map tile i-1.  Returns false if the slot is unused.
__device__ __forceinline__ bool decode_tile(const DecodeArgs& a, int slot, int& expert, int& row0,
                                            int& rows) {
  const int P = a.T * a.k;
  if (slot == 0) {
    expert = a.E;
    row0 = P;
    rows = a.T;
    return true;
  }
  const int ti = slot - 1;
  if (ti >= *a.n_tiles) return false;
  expert = a.block_map[2 * ti];
  row0 = a.block_map[2 * ti + 1];
  if (expert < 0 || expert >= a.E || row0 < 0 || row0 >= P) {
    if (threadIdx.x == 0) set_status(a.status, LILY_STATUS_BAD_TILE);
    return false;
  }
  rows = min(kDecMaxRows, a.offsets[expert + 1] - row0);
  return rows > 0;
}

// Activation rows -> shared memory in the permuted pair order, plus the
// per-group sums X_g.  src(n, i) gives the 16-bit pattern of element i of
// row n (n < rows), bf16 or fp16 as F16 says.
//   xp[(n*G + g)*32 + c*8 + w*4 + m*2 + r] =
//     (x[n][g*64 + c*16 + 8w + 2m + r], x[n][... + 4])
template <bool F16, typename Src>
__device__ void stage_rows(uint32_t* xp, float* xs, int rows, int K, Src src) {
  const int G = K / 64;
  const int total = kDecMaxRows * G * 32;
  for (int e = threadIdx.x; e < total; e += kDecThreads) {
    const int n = e / (G * 32), rem = e % (G * 32), g = rem / 32, idx = rem % 32;
    const int c = idx >> 3, w = (idx >> 2) & 1, m = (idx >> 1) & 1, r = idx & 1;
    uint32_t v = 0;
    if (n < rows) {
      const int i = g * 64 + c * 16 + 8 * w + 2 * m + r;
      v = (uint32_t)src(n, i) | ((uint32_t)src(n, i + 4) << 16);
    }
    xp[e] = v;
  }
  __syncthreads();
  // group sums from the staged copy (shared memory), not from global memory
  for (int e = threadIdx.x; e < kDecMaxRows * G; e += kDecThreads) {
    const int n = e / G;
    float s = 0.f;
    if (n < rows) {
      const uint32_t* p = xp + (size_t)e * 32;
#pragma unroll 8
      for (int i = 0; i < 32; ++i) {
        const uint32_t v = p[i];
        s += act_to_float<F16>((uint16_t)(v & 0xFFFFu)) + act_to_float<F16>((uint16_t)(v >> 16));
      }
    }
    xs[e] = s;
  }
}

// 16 weight rows [r0, r0+16) of one packed matrix (row length K) times the
// staged activations, over the groups g = g_begin, g_begin + g_step, ...
// Accumulates into out[4] = (row g, tok 2c), (g, 2c+1), (g+8, 2c), (g+8, 2c+1).
template <bool F16>
__device__ __forceinline__ void gemv16(const uint8_t* __restrict__ q, const uint16_t* __restrict__ s,
                                       const uint16_t* __restrict__ b, size_t r0, int K,
                                       const uint32_t* xp, const float* xs, int g_begin,
                                       int g_step, float (&out)[4]) {
  const int lane = threadIdx.x & 31, gi = lane >> 2, c = lane & 3;
  const int G = K / 64;
  const uint8_t* qa = q + (r0 + gi) * (size_t)(K / 2) + c * 8;
  const uint8_t* qb = qa + 8 * (size_t)(K / 2);
  const uint16_t* sa = s + (r0 + gi) * (size_t)G;
  const uint16_t* sb_ = sa + 8 * (size_t)G;
  const uint16_t* ba = b + (r0 + gi) * (size_t)G;
  const uint16_t* bb = ba + 8 * (size_t)G;
  for (int g = g_begin; g < G; g += g_step) {
    const uint2 wa = __ldcs(reinterpret_cast<const uint2*>(qa + g * 32));
    const uint2 wb = __ldcs(reinterpret_cast<const uint2*>(qb + g * 32));
    const float s_a = bf16_bits_to_float(__ldg(sa + g)), s_b = bf16_bits_to_float(__ldg(sb_ + g));
    const float b_a = bf16_bits_to_float(__ldg(ba + g)), b_b = bf16_bits_to_float(__ldg(bb + g));
    const uint32_t* xg = xp + ((size_t)gi * G + g) * 32 + c * 8;  // token n = gi for B
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      uint32_t pa[4], pb[4];
      code_pairs<F16>(w == 0 ? wa.x : wa.y, pa);
      code_pairs<F16>(w == 0 ? wb.x : wb.y, pb);
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const uint32_t afrag[4] = {pa[2 * m], pb[2 * m], pa[2 * m + 1], pb[2 * m + 1]};
        mma_16816<F16>(acc, afrag, xg[w * 4 + m * 2], xg[w * 4 + m * 2 + 1]);
      }
    }
    constexpr float off = F16 ? 1024.f : 128.f;  // the code offset of the magic
    const float x0 = xs[(2 * c) * G + g], x1 = xs[(2 * c + 1) * G + g];
    out[0] += s_a * (acc[0] - off * x0) + b_a * x0;
    out[1] += s_a * (acc[1] - off * x1) + b_a * x1;
    out[2] += s_b * (acc[2] - off * x0) + b_b * x0;
    out[3] += s_b * (acc[3] - off * x1) + b_b * x1;
  }
}

// Gate/up: CTA = (tile slot, 16 features); 8 warps split K; H = silu(g) * u.
__global__ void __launch_bounds__(kDecThreads) dec_gateup_kernel(const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const int G = a.d / 64;
  uint32_t* xp = reinterpret_cast<uint32_t*>(smem_raw);    // [8][G][32]
  float* xs = reinterpret_cast<float*>(xp + kDecMaxRows * G * 32);  // [8][G]
  float* part = xs + kDecMaxRows * G;                      // [8 warps][2][16][8]
  __shared__ int tok[kDecMaxRows];

  const int nfb = a.F / 16;
  const int slot = blockIdx.x / nfb, fb = blockIdx.x % nfb;
  int expert, row0, rows;
  if (!decode_tile(a, slot, expert, row0, rows)) return;
  const int P = a.T * a.k;
  if (threadIdx.x < kDecMaxRows) {
    const int n = min((int)threadIdx.x, rows - 1);
    tok[threadIdx.x] = (slot == 0) ? n : a.perm[row0 + n] / a.k;
  }
  __syncthreads();
  const uint16_t* x = static_cast<const uint16_t*>(a.x);
  stage_rows<false>(xp, xs, rows, a.d, [&](int n, int i) { return x[(size_t)tok[n] * a.d + i]; });
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t r0 = (size_t)expert * a.F + (size_t)fb * 16;
  float og[4] = {0.f, 0.f, 0.f, 0.f}, ou[4] = {0.f, 0.f, 0.f, 0.f};
  gemv16<false>(a.gq, a.gs, a.gb, r0, a.d, xp, xs, warp, 8, og);
  gemv16<false>(a.uq, a.us, a.ub, r0, a.d, xp, xs, warp, 8, ou);
  {
    const int gi = lane >> 2, c = lane & 3;
    float* pw = part + warp * 256;
    pw[0 * 128 + gi * 8 + 2 * c] = og[0];
    pw[0 * 128 + gi * 8 + 2 * c + 1] = og[1];
    pw[0 * 128 + (gi + 8) * 8 + 2 * c] = og[2];
    pw[0 * 128 + (gi + 8) * 8 + 2 * c + 1] = og[3];
    pw[1 * 128 + gi * 8 + 2 * c] = ou[0];
    pw[1 * 128 + gi * 8 + 2 * c + 1] = ou[1];
    pw[1 * 128 + (gi + 8) * 8 + 2 * c] = ou[2];
    pw[1 * 128 + (gi + 8) * 8 + 2 * c + 1] = ou[3];
  }
  __syncthreads();
  if (threadIdx.x < 128) {
    const int t = threadIdx.x;  // (row, token) = (t / 8, t % 8)
    float g = 0.f, u = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      g += part[w * 256 + t];
      u += part[w * 256 + 128 + t];
    }
    const int row = t >> 3, n = t & 7;
    if (n < rows) {
      const float h = g / (1.f + __expf(-g)) * u;
      if (!(fabsf(h) <= 65504.f)) set_status(a.status, LILY_STATUS_F16_RANGE);
      static_cast<__half*>(a.H)[(size_t)(row0 + n) * a.F + fb * 16 + row] = __float2half_rn(h);
    }
  }
  (void)P;
}

// Down: CTA = (tile slot, 128 output features); each warp owns 16 features
// over all of K = F.  Writes O[row][feature] (fp32, expert-sorted rows).
__global__ void __launch_bounds__(kDecThreads) dec_down_kernel(const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const int G = a.F / 64;
  uint32_t* xp = reinterpret_cast<uint32_t*>(smem_raw);
  float* xs = reinterpret_cast<float*>(xp + kDecMaxRows * G * 32);

  const int nob = a.d / 128;
  const int slot = blockIdx.x / nob, ob = blockIdx.x % nob;
  int expert, row0, rows;
  if (!decode_tile(a, slot, expert, row0, rows)) return;
  const uint16_t* H = static_cast<const uint16_t*>(a.H);
  stage_rows<true>(xp, xs, rows, a.F, [&](int n, int i) { return H[(size_t)(row0 + n) * a.F + i]; });
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int feat0 = ob * 128 + warp * 16;
  float o[4] = {0.f, 0.f, 0.f, 0.f};
  gemv16<true>(a.dq, a.ds, a.db, (size_t)expert * a.d + feat0, a.F, xp, xs, 0, 1, o);
  const int gi = lane >> 2, c = lane & 3;
  const int n0 = 2 * c, n1 = 2 * c + 1;
  if (n0 < rows) {
    a.O[(size_t)(row0 + n0) * a.d + feat0 + gi] = o[0];
    a.O[(size_t)(row0 + n0) * a.d + feat0 + gi + 8] = o[2];
  }
  if (n1 < rows) {
    a.O[(size_t)(row0 + n1) * a.d + feat0 + gi] = o[1];
    a.O[(size_t)(row0 + n1) * a.d + feat0 + gi + 8] = o[3];
  }
}

// y[t] = sum_j gate[t][j] * O[inv[t*k+j]] + O[P + t], in slot order (fp32,
// or rounded once to bf16).  Grid: (T, d / 256).
__global__ void __launch_bounds__(256) dec_combine_kernel(const DecodeArgs a) {
  const int t = blockIdx.x;
  const int P = a.T * a.k;
  for (int i = blockIdx.y * blockDim.x + threadIdx.x; i < a.d; i += gridDim.y * blockDim.x) {
    float acc = 0.f;
    for (int j = 0; j < a.k; ++j) {
      const int p = t * a.k + j;
      acc += a.gates[p] * a.O[(size_t)a.inv[p] * a.d + i];
    }
    acc += a.O[(size_t)(P + t) * a.d + i];
    if (a.y_f32)
      static_cast<float*>(a.y)[(size_t)t * a.d + i] = acc;
    else
      static_cast<__nv_bfloat16*>(a.y)[(size_t)t * a.d + i] = __float2bfloat16_rn(acc);
  }
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  if (a.T < 1 || a.T > kDecMaxRows) return cudaErrorInvalidValue;
  const int slots = 1 + a.cap;
  const size_t smem_gu = (size_t)kDecMaxRows * (a.d / 64) * (32 * 4 + 4) + 8 * 256 * 4;
  const size_t smem_dn = (size_t)kDecMaxRows * (a.F / 64) * (32 * 4 + 4);
  cudaError_t err;
  if ((err = ensure_smem_attr((const void*)dec_gateup_kernel, smem_gu)) != cudaSuccess) return err;
  if ((err = ensure_smem_attr((const void*)dec_down_kernel, smem_dn)) != cudaSuccess) return err;
  prof_begin(K_DEC_GATEUP, s);
  dec_gateup_kernel<<<slots * (a.F / 16), kDecThreads, smem_gu, s>>>(a);
  prof_end(K_DEC_GATEUP, s);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  prof_begin(K_DEC_DOWN, s);
  dec_down_kernel<<<slots * (a.d / 128), kDecThreads, smem_dn, s>>>(a);
  prof_end(K_DEC_DOWN, s);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  prof_begin(K_DEC_COMBINE, s);
  dec_combine_kernel<<<dim3(a.T, (a.d + 255) / 256), 256, 0, s>>>(a);
  prof_end(K_DEC_COMBINE, s);
  return cudaGetLastError();
}

}  // namespace lily
