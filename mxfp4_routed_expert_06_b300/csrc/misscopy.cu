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
__device__ __forceinline__ void copy_misses(const MissCopy* __restrict__ list, int n, size_t bytes) {
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

// The miss list and its count come from the host bookkeeping (kernel arguments).
__global__ void __launch_bounds__(kMcThreads) miss_copy_kernel(const MissCopy* __restrict__ list, int n,
                                                               size_t bytes) {
  copy_misses(list, n, bytes);
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

// ------------------------------------------------------------- device-side LRU lookup ---
// The expert cache with its LRU state on the device (k3moe_cache_set_device_lru): a layer call
// looks its active experts up with one thread, on its own stream, right after routing, so that
// no host round trip sits between routing and the FFN.  The policy is the host bookkeeping's:
// the call's hits are made most recently used first (in active-list order), then each miss takes
// the least recently used slot (which the call cannot be using: it needs at most n_slots
// experts, checked when the layer attaches) and is listed for the copy kernel below.
namespace k3 {
namespace {

__device__ __forceinline__ void lru_unlink(LruState* st, int32_t* prev, int32_t* next, int s) {
  const int p = prev[s], n = next[s];
  if (p >= 0) next[p] = n; else st->head = n;
  if (n >= 0) prev[n] = p; else st->tail = p;
}
__device__ __forceinline__ void lru_push_front(LruState* st, int32_t* prev, int32_t* next, int s) {
  prev[s] = -1;
  next[s] = st->head;
  if (st->head >= 0) prev[st->head] = s; else st->tail = s;
  st->head = s;
}
__device__ __forceinline__ void lru_push_back(LruState* st, int32_t* prev, int32_t* next, int s) {
  next[s] = -1;
  prev[s] = st->tail;
  if (st->tail >= 0) next[st->tail] = s; else st->head = s;
  st->tail = s;
}

__global__ void lru_lookup_kernel(LruArgs a) {
  pdl_entry();
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  LruState* st = a.state;
  const int nact = *a.nact;
  int nm = 0;
  if (nact < 0 || nact > a.n_slots) {  // cannot happen for an attached layer; leave the pointers alone
    atomicOr(a.err, kErrBudget);
    *a.nmiss = 0;
    return;
  }
  for (int i = 0; i < nact; ++i) {  // hits first
    const int e = a.act[i];
    const int s = a.slot_of[e];
    if (s >= 0) {
      lru_unlink(st, a.prev, a.next, s);
      lru_push_front(st, a.prev, a.next, s);
      a.eptr[e] = a.slots + (size_t)s * a.slot_bytes;
      st->hits += 1;
    }
  }
  for (int i = 0; i < nact; ++i) {  // then the misses, each into the least recently used slot
    const int e = a.act[i];
    if (a.slot_of[e] >= 0) continue;
    const int s = st->tail;
    lru_unlink(st, a.prev, a.next, s);
    if (a.owner[s] != nullptr) {
      *a.owner[s] = -1;
      st->evictions += 1;
    }
    a.owner[s] = a.slot_of + e;
    a.slot_of[e] = s;
    lru_push_front(st, a.prev, a.next, s);
    uint8_t* dst = a.slots + (size_t)s * a.slot_bytes;
    a.eptr[e] = dst;
    a.miss[nm++] = MissCopy{a.pool_dev + (size_t)e * a.slot_bytes, dst};
    st->misses += 1;
  }
  st->calls += 1;
  *a.nmiss = nm;
}

// A layer leaves the cache: the slots it owns become empty and least recently used.
__global__ void lru_detach_kernel(LruState* st, int32_t* prev, int32_t* next, int32_t** owner, int n_slots,
                                  const int32_t* slot_of, int E) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  for (int s = 0; s < n_slots; ++s) {
    if (owner[s] != nullptr && owner[s] >= slot_of && owner[s] < slot_of + E) {
      owner[s] = nullptr;
      lru_unlink(st, prev, next, s);
      lru_push_back(st, prev, next, s);
    }
  }
}

// The copy kernel for a miss list and count written on the device by the lookup kernel.
__global__ void __launch_bounds__(kMcThreads) miss_copy_dev_kernel(const MissCopy* __restrict__ list,
                                                                   const int32_t* n_dev, size_t bytes) {
  pdl_entry();
  copy_misses(list, *n_dev, bytes);
}

}  // namespace

cudaError_t launch_lru_lookup(const LruArgs& a, cudaStream_t s) {
  return launch_pdl(lru_lookup_kernel, dim3(1), dim3(32), 0, s, a);
}

cudaError_t launch_miss_copy_dev(const MissCopy* list, const int32_t* n_dev, int max_n, size_t bytes, int num_sms,
                                 cudaStream_t s) {
  const size_t chunks = (bytes + kMcChunk - 1) / kMcChunk * (size_t)(max_n > 0 ? max_n : 1);
  const int grid = (int)(chunks < (size_t)num_sms * 4 ? chunks : (size_t)num_sms * 4);
  return launch_pdl(miss_copy_dev_kernel, dim3(grid), dim3(kMcThreads), 0, s, list, n_dev, bytes);
}

cudaError_t launch_lru_detach(LruState* st, int32_t* prev, int32_t* next, int32_t** owner, int n_slots,
                              const int32_t* slot_of, int E, cudaStream_t s) {
  lru_detach_kernel<<<1, 32, 0, s>>>(st, prev, next, owner, n_slots, slot_of, E);
  return cudaGetLastError();
}

}  // namespace k3
