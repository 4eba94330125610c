// Glue between stacked MoE layers: residual add and a weightless RMSNorm.
//
// The layer's output excludes the residual.  A caller that stacks layers adds each output to
// its input, x_next = bf16_rne(x + y) with the sum in fp32, and feeds the next layer the
// RMSNorm of that sum, x_norm = bf16_rne(x_next / sqrt(mean(x_next^2) + eps)), as a pre-norm
// transformer block does (the kimi-k3-in-c deep dive, "what you learn", names the engine's
// RMSNorm kernel).  One CTA per token; HBM-bound and tiny (d = 7168: 14 KB in, 28 KB out).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "k3moe_internal.cuh"

namespace k3 {
namespace {

constexpr int kGlueThreads = 256;

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ uint16_t float_to_bf16_bits(float v) {
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  return *reinterpret_cast<const uint16_t*>(&h);
}

__global__ void __launch_bounds__(kGlueThreads) residual_rmsnorm_kernel(const float* __restrict__ y,
                                                                        const uint16_t* x, int d, float eps,
                                                                        uint16_t* x_next, uint16_t* x_norm) {
  __shared__ float part[kGlueThreads / 32];
  pdl_entry();
  const size_t base = (size_t)blockIdx.x * d;
  float ss = 0.f;
  // each thread owns the elements j = tid + i*blockDim; it reads back only its own writes
  for (int j = threadIdx.x; j < d; j += kGlueThreads) {
    const float r = bf16_bits_to_float(float_to_bf16_bits(bf16_bits_to_float(x[base + j]) + y[base + j]));
    x_next[base + j] = float_to_bf16_bits(r);
    ss = fmaf(r, r, ss);
  }
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kGlueThreads / 32; ++w) tot += part[w];
  const float inv = 1.0f / sqrtf(tot / (float)d + eps);
  for (int j = threadIdx.x; j < d; j += kGlueThreads)
    x_norm[base + j] = float_to_bf16_bits(bf16_bits_to_float(x_next[base + j]) * inv);
}

}  // namespace

cudaError_t launch_residual_rmsnorm(const float* y, const uint16_t* x, int T, int d, float eps, uint16_t* x_next,
                                    uint16_t* x_norm, cudaStream_t s) {
  return launch_pdl(residual_rmsnorm_kernel, dim3(T), dim3(kGlueThreads), 0, s, y, x, d, eps, x_next, x_norm);
}

}  // namespace k3
