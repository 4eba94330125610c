// k3synth_dev.cu -- device side of the counter-based synthetic-input generator.
//
// Fills canonical MXFP4 expert bytes straight into device memory, so that a
// 15.7 GB layer does not have to be generated on the host and copied.  Only the
// integer streams (tags 1 and 2 of k3synth.h) exist here; they are bit-identical
// to the host functions by construction (same 64-bit integer arithmetic).
#include <cstdint>
#include <cuda_runtime.h>
#include "k3synth.h"

namespace {

__device__ __forceinline__ uint64_t dmix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

__global__ void gen_nibbles(uint64_t seed, uint32_t layer, int e0, int nexp, uint64_t mat_words, uint8_t* nib) {
  const uint64_t total = (uint64_t)nexp * 3 * mat_words;
  for (uint64_t w = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; w < total;
       w += (uint64_t)gridDim.x * blockDim.x) {
    const uint64_t em = w / mat_words, i = w % mat_words;
    const uint32_t e = (uint32_t)(e0 + em / 3), m = (uint32_t)(em % 3);
    const uint64_t key = k3s_key(seed, K3S_TAG_NIB, layer, e, m);
    reinterpret_cast<uint64_t*>(nib)[w] = dmix(key + (i + 1) * K3S_GAMMA);
  }
}

__global__ void gen_scales(uint64_t seed, uint32_t layer, int e0, int nexp, uint64_t mat_scl, int lo, int hi,
                           uint8_t* scl) {
  const uint64_t total = (uint64_t)nexp * 3 * mat_scl;
  const uint64_t r = (uint64_t)(hi - lo + 1);
  for (uint64_t j = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; j < total;
       j += (uint64_t)gridDim.x * blockDim.x) {
    const uint64_t em = j / mat_scl, i = j % mat_scl;
    const uint32_t e = (uint32_t)(e0 + em / 3), m = (uint32_t)(em % 3);
    const uint64_t key = k3s_key(seed, K3S_TAG_SCALE, layer, e, m);
    scl[j] = (uint8_t)(lo + (int)(((dmix(key + (i + 1) * K3S_GAMMA) >> 32) * r) >> 32));
  }
}

}  // namespace

extern "C" int k3s_dev_experts(uint64_t seed, int layer, int e0, int e1, int d, int f, int scale_lo, int scale_hi,
                               void* nib_dev, void* scl_dev, void* stream) {
  if (e1 <= e0 || d <= 0 || f <= 0 || ((size_t)f * d) % 32 != 0) return -1;
  if (((uintptr_t)nib_dev & 7) != 0) return -1;
  const int nexp = e1 - e0;
  const uint64_t mat_words = (uint64_t)f * d / 16, mat_scl = (uint64_t)f * d / 32;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  gen_nibbles<<<148 * 16, 256, 0, s>>>(seed, (uint32_t)layer, e0, nexp, mat_words, (uint8_t*)nib_dev);
  gen_scales<<<148 * 16, 256, 0, s>>>(seed, (uint32_t)layer, e0, nexp, mat_scl, scale_lo, scale_hi,
                                       (uint8_t*)scl_dev);
  return cudaGetLastError() == cudaSuccess ? 0 : -2;
}
