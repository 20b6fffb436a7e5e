// misc.cu -- unit-weight RMSNorm, the pre-norm of the stacked-layer prefill
// (the residual add and the next layer's norm are fused into the combine).
//
// The pages name no normalisation around the MoE block; a bare residual stack
// x <- x + MoE(x) of SwiGLU experts grows without bound, so the stack uses the
// standard pre-norm block x <- x + MoE(bf16(rmsnorm(x))) with an fp32
// residual to which the layer's fp32 output is added.  Long prompts run in bounded chunks (page "Lily Beats MLX-LM
// 1.35x on Decode: Perplexity's Rust+Metal Engine for Apple Silicon", section
// "Prefill: fusing dequantisation and keeping routing GPU-resident").
#include "common.cuh"

namespace lily {

constexpr int kRowThreads = 256;

__device__ float block_sum(float v, float* tmp /* [8] */) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) tmp[warp] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int w = 0; w < kRowThreads / 32; ++w) s += tmp[w];
  __syncthreads();
  return s;
}

__device__ void rms_row(const float* xr, __nv_bfloat16* outr, int d, float eps, float* tmp) {
  float ss = 0.f;
  for (int i = threadIdx.x; i < d; i += kRowThreads) ss += xr[i] * xr[i];
  const float tot = block_sum(ss, tmp);
  const float inv = 1.f / sqrtf(tot / (float)d + eps);
  for (int i = threadIdx.x; i < d; i += kRowThreads) outr[i] = __float2bfloat16_rn(xr[i] * inv);
}

__global__ void __launch_bounds__(kRowThreads) rmsnorm_kernel(const float* __restrict__ x,
                                                              __nv_bfloat16* __restrict__ out,
                                                              int d, float eps) {
  __shared__ float tmp[8];
  const size_t row = blockIdx.x;
  rms_row(x + row * d, out + row * d, d, eps, tmp);
}

cudaError_t launch_rmsnorm(const float* x, void* out, int T, int d, float eps, cudaStream_t s) {
  prof_begin(K_RMSNORM, s);
  rmsnorm_kernel<<<T, kRowThreads, 0, s>>>(x, static_cast<__nv_bfloat16*>(out), d, eps);
  prof_end(K_RMSNORM, s);
  return cudaGetLastError();
}

}  // namespace lily
