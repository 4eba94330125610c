// noalloc.cu -- router + top-k for callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc: code embedded in a host framework whose memory pool
// already owns the device memory (a further cudaMalloc can fail, or break the framework's
// accounting), and latency-critical loops where an allocation may implicitly synchronise the
// device.  Creating a layer object allocates (packed weights, workspace), so
// k3moe_router_topk_noalloc takes every input and output from the caller and keeps its only
// scratch -- the router logits between the GEMV phase and the top-k phase, and the ticket
// that elects the last block -- in one file-scope device array of fixed size.
//
// Set-up: the first call on a device (with that device current) resolves the array's device
// address with cudaGetSymbolAddress; later calls on that device reuse it.  The scratch is
// shared by every call on a device and keeps the last call's contents: the ticket is cleared
// on the stream before each launch, the logits are fully rewritten.  Calls that overlap on the
// GPU (two streams at once) race on the scratch.
#include <mutex>

#include "k3moe_internal.cuh"

namespace {

constexpr size_t kMaxLogits = 65536;                    // T * E <= 65536
constexpr size_t kTicketBytes = 256;                    // [0, 256): last-block ticket
constexpr size_t kScratchBytes = kTicketBytes + kMaxLogits * sizeof(float);  // 256 KiB + 256 B

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kWarps = 4;
constexpr int kTok = 4;

int fail(int code, const char* msg) {
  k3::set_last_error(msg);
  return code;
}

__device__ __forceinline__ float sig(float z) { return 1.0f / (1.0f + expf(-z)); }

// A float's bits as an unsigned integer with the same order (larger float -> larger integer);
// NaNs land at the two ends according to their sign bit.
__device__ __forceinline__ uint32_t ord_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(kWarps * 32) router_topk_noalloc_kernel(
    const uint16_t* __restrict__ x, const float* __restrict__ Wr, const float* __restrict__ bias, int T, int d, int E,
    int k, int32_t* __restrict__ idx, float* __restrict__ w, unsigned char* scratch) {
  extern __shared__ unsigned long long keys[];  // [kWarps][E] rank keys of the last block
  __shared__ int last;
  unsigned int* ticket = reinterpret_cast<unsigned int*>(scratch);
  float* logits = reinterpret_cast<float*>(scratch + kTicketBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * kWarps + warp;
  if (e < E) {
    const float4* wr = reinterpret_cast<const float4*>(Wr + (size_t)e * d);
    for (int t0 = 0; t0 < T; t0 += kTok) {
      float acc[kTok] = {0.f, 0.f, 0.f, 0.f};
      const int nt = min(kTok, T - t0);
      for (int q = lane; q < d / 4; q += 32) {
        const float4 wv = __ldg(wr + q);
#pragma unroll
        for (int tt = 0; tt < kTok; ++tt) {
          if (tt < nt) {
            const uint2 xv = __ldg(reinterpret_cast<const uint2*>(x + (size_t)(t0 + tt) * d) + q);
            acc[tt] = fmaf(__uint_as_float(xv.x << 16), wv.x, acc[tt]);
            acc[tt] = fmaf(__uint_as_float(xv.x & 0xFFFF0000u), wv.y, acc[tt]);
            acc[tt] = fmaf(__uint_as_float(xv.y << 16), wv.z, acc[tt]);
            acc[tt] = fmaf(__uint_as_float(xv.y & 0xFFFF0000u), wv.w, acc[tt]);
          }
        }
      }
#pragma unroll
      for (int tt = 0; tt < kTok; ++tt) {
        float v = acc[tt];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == 0 && tt < nt) logits[(size_t)(t0 + tt) * E + e] = v;
      }
    }
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = (atomicAdd(ticket, 1u) == gridDim.x - 1);
  __syncthreads();
  if (!last) return;
  __threadfence();
  // Top-k per token, one warp per token.  Every expert j gets the 64-bit rank key
  //   (order-preserving bits of sigma + bias) << 32  |  ~j
  // so a larger rank key means a larger selection key, or an equal one and a lower expert id:
  // the same total order as k3moe_router_topk, NaN and infinite keys included.  Every real
  // entry's rank key is nonzero (its low word ~j is), and a picked entry is set to 0, so the
  // warp-wide maximum of each of the k rounds is always an entry not yet picked: every selected
  // id lies in 0..E-1 whatever the key values (E >= k is checked on the host).
  unsigned long long* ks = keys + (size_t)warp * E;
  for (int t = warp; t < T; t += kWarps) {
    const float* row = logits + (size_t)t * E;
    for (int j0 = 0; j0 < E; j0 += 32 * 16) {  // 16 loads in flight per lane
      float z[16], bb[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const int j = j0 + 32 * q + lane;
        z[q] = j < E ? __ldcg(row + j) : 0.f;
        bb[q] = (bias && j < E) ? __ldg(bias + j) : 0.f;
      }
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const int j = j0 + 32 * q + lane;
        if (j < E) ks[j] = ((unsigned long long)ord_key(sig(z[q]) + bb[q]) << 32) | (unsigned long long)(~(uint32_t)j);
      }
    }
    __syncwarp();
    int mine = -1;
    for (int i = 0; i < k; ++i) {
      unsigned long long best = 0ull;
      for (int j = lane; j < E; j += 32) {
        const unsigned long long c = ks[j];
        best = c > best ? c : best;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
        best = o > best ? o : best;
      }
      const int bi = (int)(~(uint32_t)(best & 0xffffffffull));
      if (lane == i) mine = bi;
      __syncwarp();
      if (lane == 0 && best != 0ull && bi >= 0 && bi < E) ks[bi] = 0ull;
      __syncwarp();
    }
    const bool ok = lane < k && mine >= 0 && mine < E;
    const float s = ok ? sig(__ldcg(row + mine)) : 0.f;
    float tot = s;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
    if (lane < k) {
      idx[(size_t)t * k + lane] = mine;
      w[(size_t)t * k + lane] = s / tot;
    }
    __syncwarp();
  }
  if (threadIdx.x == 0) *ticket = 0u;
}

struct DeviceScratch {
  void* ptr = nullptr;
  bool ready = false;
};
std::mutex g_lock;
DeviceScratch g_dev[64];

// Resolve (once per device, with that device current) the device address of the scratch array.
int scratch_for_current_device(unsigned char** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
    return fail(K3MOE_ERR_CUDA, "no current CUDA device");
  std::lock_guard<std::mutex> g(g_lock);
  if (!g_dev[dev].ready) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return fail(K3MOE_ERR_CUDA, (std::string("cudaGetSymbolAddress(no-alloc scratch): ") + cudaGetErrorString(e)).c_str());
    cudaError_t a = cudaFuncSetAttribute(router_topk_noalloc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kWarps * 4096 * (int)sizeof(unsigned long long));
    if (a != cudaSuccess) return fail(K3MOE_ERR_CUDA, (std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(a)).c_str());
    g_dev[dev].ptr = p;
    g_dev[dev].ready = true;
  }
  *out = static_cast<unsigned char*>(g_dev[dev].ptr);
  return K3MOE_OK;
}

}  // namespace

extern "C" int k3moe_router_topk_noalloc(const void* x_bf16, const float* W_r, const float* bias, int T, int d, int E,
                                         int k, int32_t* idx, float* w, void* stream) {
  if (!x_bf16 || !W_r || !idx || !w) return fail(K3MOE_ERR_INVALID_ARG, "NULL argument");
  if (d < 4 || d % 4 != 0) return fail(K3MOE_ERR_INVALID_ARG, "d must be a positive multiple of 4");
  if (E < 1 || E > 4096) return fail(K3MOE_ERR_INVALID_ARG, "E must be in 1..4096");
  if (k < 1 || k > E || k > 32) return fail(K3MOE_ERR_INVALID_ARG, "k must be in 1..min(E, 32)");
  if (T < 1) return fail(K3MOE_ERR_INVALID_ARG, "T must be >= 1");
  if ((size_t)T * (size_t)E > kMaxLogits)
    return fail(K3MOE_ERR_INVALID_ARG, "T*E exceeds the no-alloc scratch limit of 65536 router logits");
  if (!k3::aligned_to(x_bf16, 8) || !k3::aligned_to(W_r, 16))
    return fail(K3MOE_ERR_INVALID_ARG, "x must be 8-byte and W_r 16-byte aligned");
  if (!k3::aligned_to(idx, 4) || !k3::aligned_to(w, 4) || (bias && !k3::aligned_to(bias, 4)))
    return fail(K3MOE_ERR_INVALID_ARG, "idx, w and bias must be 4-byte aligned");
  unsigned char* scratch = nullptr;
  int rc = scratch_for_current_device(&scratch);
  if (rc) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, sizeof(unsigned int), s) != cudaSuccess)
    return fail(K3MOE_ERR_CUDA, "clearing the no-alloc ticket failed");
  const int grid = (E + kWarps - 1) / kWarps;
  router_topk_noalloc_kernel<<<grid, kWarps * 32, (size_t)kWarps * E * sizeof(unsigned long long), s>>>(
      reinterpret_cast<const uint16_t*>(x_bf16), W_r, bias, T, d, E, k, idx, w, scratch);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(K3MOE_ERR_CUDA, (std::string("router_topk_noalloc launch: ") + cudaGetErrorString(e)).c_str());
  return K3MOE_OK;
}
