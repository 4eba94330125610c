// misscopy.cu -- the expert cache's zero-copy miss path (K3MOE_MISS_ZERO_COPY).
//
// "kimi-k3-in-c deep dive", "four reductions", expert LRU paragraph: an LRU expert cache with
// batch prefetch.  Here a missed expert is not handed to a copy engine one cudaMemcpyAsync at a
// time: after the host's LRU bookkeeping, one kernel launch on the layer's stream copies every
// expert the call missed, the SMs reading the mapped pinned pool straight over the host link
// with 16-byte loads and writing each expert into its device slot.  The FFN kernels then read
// the slots as on a hit, so the arithmetic (and the output) does not change.
#include "k3moe_internal.cuh"

namespace k3 {
namespace {

constexpr int kMcThreads = 256;
constexpr int kMcUnroll = 4;                                           // loads in flight per thread
constexpr size_t kMcChunk = (size_t)kMcThreads * kMcUnroll * 16 * 4;   // 64 KB per CTA step

// CTA b copies chunks b, b + gridDim.x, ... of the concatenation of the n missed experts
// (`bytes` each, a multiple of 16; both addresses 16-byte aligned).
__global__ void __launch_bounds__(kMcThreads) miss_copy_kernel(const MissCopy* __restrict__ list, int n,
                                                               size_t bytes) {
  const size_t per = (bytes + kMcChunk - 1) / kMcChunk;
  const size_t total = per * (size_t)n;
  for (size_t c = blockIdx.x; c < total; c += gridDim.x) {
    const int m = (int)(c / per);
    const size_t base = (c % per) * kMcChunk;
    const uint4* src = reinterpret_cast<const uint4*>(list[m].src + base);
    uint4* dst = reinterpret_cast<uint4*>(list[m].dst + base);
    const size_t words = (bytes - base < kMcChunk ? bytes - base : kMcChunk) / 16;
    for (size_t w0 = threadIdx.x; w0 < words; w0 += (size_t)kMcThreads * kMcUnroll) {
      uint4 v[kMcUnroll];
#pragma unroll
      for (int u = 0; u < kMcUnroll; ++u) {
        const size_t w = w0 + (size_t)u * kMcThreads;
        if (w < words) v[u] = src[w];
      }
#pragma unroll
      for (int u = 0; u < kMcUnroll; ++u) {
        const size_t w = w0 + (size_t)u * kMcThreads;
        if (w < words) dst[w] = v[u];
      }
    }
  }
}

}  // namespace

cudaError_t launch_miss_copy(const MissCopy* list, int n, size_t bytes, int num_sms, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const size_t chunks = (bytes + kMcChunk - 1) / kMcChunk * (size_t)n;
  const int grid = (int)(chunks < (size_t)num_sms * 4 ? chunks : (size_t)num_sms * 4);
  miss_copy_kernel<<<grid, kMcThreads, 0, s>>>(list, n, bytes);
  return cudaGetLastError();
}

}  // namespace k3
