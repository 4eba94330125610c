// router.cu -- router logits, sigmoid + bias top-k selection, and token-to-expert bucketing.
//
// Routing rule ("kimi-k3-in-c deep dive": "what you learn", router paragraph, and the
// invariants table, row 5): sigmoid scores; the bias steers the selection only; the picked
// experts are mixed with weights from the unbiased scores, renormalised to sum 1.  The pages
// pick 16 of 896 experts (glossary entry MoE).
//
// GPU design: the router is a GEMV over W_r (fp32, [E][d]) with one warp per expert row and
// the tokens in tiles of 4, so W_r is read once per call (it stays in L2 across calls).  For
// small T the last CTA to finish (atomic ticket) also runs the top-k and the bucketing, which
// saves two launches on the single-token path.  Top-k is a warp per token: k rounds of a
// warp-wide (key desc, id asc) argmax over the keys kept in shared memory.  Bucketing is
// deterministic: counts by shared-memory atomics (order-free), an exclusive scan, and a
// stable scatter in rounds where __match_any_sync ranks equal experts inside a warp and the
// warps of a round take their turn in order.
#include "k3moe_internal.cuh"

namespace k3 {
namespace {

constexpr int kRouterWarps = 4;  // expert rows per CTA, one per warp
constexpr int kTokTile = 4;

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ float sigmoidf_acc(float z) { return 1.0f / (1.0f + expf(-z)); }

// power-of-two scale 2^q for the fp16 image of a row whose largest magnitude is m:
// m * 2^-q lies in [2^14, 2^15), so the fp16 image never overflows and keeps bf16 values exact.
__device__ __forceinline__ int fp16_scale_exp(float m) {
  if (!(m > 0.0f)) return 0;
  int ex = (int)((__float_as_uint(m) >> 23) & 0xFFu) - 127;
  int q = ex - 14;
  return q < -126 ? -126 : (q > 126 ? 126 : q);
}
__device__ __forceinline__ float exp2i(int q) { return __uint_as_float((uint32_t)(127 + q) << 23); }

// --------------------------------------------------------------------------- logits ---
__device__ void logits_rows(const RouterArgs& a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * kRouterWarps + warp;
  if (e >= a.E) return;
  const float4* wr = reinterpret_cast<const float4*>(a.Wr + (size_t)e * a.d);
  const int nq = a.d / 4;
  for (int t0 = 0; t0 < a.T; t0 += kTokTile) {
    float acc[kTokTile] = {0.f, 0.f, 0.f, 0.f};
    const int nt = min(kTokTile, a.T - t0);
#pragma unroll 8
    for (int q = lane; q < nq; q += 32) {
      const float4 w = __ldg(wr + q);
#pragma unroll
      for (int tt = 0; tt < kTokTile; ++tt) {
        if (tt < nt) {
          const uint2 xv = __ldg(reinterpret_cast<const uint2*>(a.x + (size_t)(t0 + tt) * a.d) + q);
          acc[tt] = fmaf(bf16_lo(xv.x), w.x, acc[tt]);
          acc[tt] = fmaf(bf16_hi(xv.x), w.y, acc[tt]);
          acc[tt] = fmaf(bf16_lo(xv.y), w.z, acc[tt]);
          acc[tt] = fmaf(bf16_hi(xv.y), w.w, acc[tt]);
        }
      }
    }
#pragma unroll
    for (int tt = 0; tt < kTokTile; ++tt) {
      float v = acc[tt];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0 && tt < nt) a.ws.logits[(size_t)(t0 + tt) * a.E + e] = v;
    }
  }
}

// x (bf16) -> fp16 B-fragment rows with a per-token power-of-two scale.
__device__ void convert_tokens(const RouterArgs& a, float* red) {
  for (int t = blockIdx.x; t < a.T; t += gridDim.x) {
    const uint16_t* xr = a.x + (size_t)t * a.d;
    float m = 0.f;
    for (int j = threadIdx.x; j < a.d; j += blockDim.x) m = fmaxf(m, fabsf(__uint_as_float((uint32_t)xr[j] << 16)));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    m = red[0];
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
    __syncthreads();
    const int q = fp16_scale_exp(m);
    const float inv = exp2i(-q);
    const int items = (a.d / 32) * 4;
    for (int it = threadIdx.x; it < items; it += blockDim.x) {
      const int blk = it >> 2, tq = it & 3;
      __align__(16) __half h[8];
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        const int kb = 32 * blk + 16 * s + 2 * tq;
        h[4 * s + 0] = __float2half_rn(__uint_as_float((uint32_t)xr[kb] << 16) * inv);
        h[4 * s + 1] = __float2half_rn(__uint_as_float((uint32_t)xr[kb + 1] << 16) * inv);
        h[4 * s + 2] = __float2half_rn(__uint_as_float((uint32_t)xr[kb + 8] << 16) * inv);
        h[4 * s + 3] = __float2half_rn(__uint_as_float((uint32_t)xr[kb + 9] << 16) * inv);
      }
      *reinterpret_cast<uint4*>(a.ws.xfrag + (size_t)t * a.d + (size_t)it * 8) = *reinterpret_cast<uint4*>(h);
    }
    if (threadIdx.x == 0) a.ws.xscale[t] = exp2i(q);
  }
}

}  // namespace

// ---------------------------------------------------------------------------- top-k ---
// One warp selects the k largest keys of one token.  ks: E floats of this warp's shared memory.
__device__ void topk_warp(const float* logits_row, const float* bias, int E, int k, float* ks, int32_t* idx_out,
                          float* w_out) {
  const int lane = threadIdx.x & 31;
  for (int e = lane; e < E; e += 32) {
    const float s = sigmoidf_acc(__ldcg(logits_row + e));
    ks[e] = bias ? s + __ldg(bias + e) : s;
  }
  __syncwarp();
  int mine = -1;
  for (int i = 0; i < k; ++i) {
    float bk = -INFINITY;
    int bi = 0x7fffffff;
    for (int e = lane; e < E; e += 32) {
      const float v = ks[e];
      if (v > bk || (v == bk && e < bi)) { bk = v; bi = e; }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ok = __shfl_xor_sync(0xffffffffu, bk, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (ok > bk || (ok == bk && oi < bi)) { bk = ok; bi = oi; }
    }
    if (lane == i) mine = bi;
    __syncwarp();
    if (lane == 0 && bi < E) ks[bi] = -INFINITY;
    __syncwarp();
  }
  const float sg = (lane < k && mine >= 0) ? sigmoidf_acc(__ldcg(logits_row + mine)) : 0.f;
  float tot = sg;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
  if (lane < k) {
    idx_out[lane] = mine;
    w_out[lane] = sg / tot;
  }
  __syncwarp();
}

// ------------------------------------------------------------------------ bucketing ---
// Whole-block deterministic bucketing of P picks.  smem: 2*E ints.
__device__ void bucket_block(const int32_t* idx, int P, int k, int E, int32_t* counts, int32_t* offsets,
                             int32_t* perm, int32_t* act, int32_t* nact, UnitDesc* units, int32_t* nunits,
                             const float* w, const float* xscale, int* smem) {
  __shared__ int s_nunits;
  int* cnt = smem;
  int* cur = smem + E;
  const int tid = threadIdx.x, bd = blockDim.x, warp = tid >> 5, lane = tid & 31, nwarps = bd >> 5;
  for (int e = tid; e < E; e += bd) cnt[e] = 0;
  __syncthreads();
  for (int p = tid; p < P; p += bd) {
    const int e = __ldcg(idx + p);
    if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  if (warp == 0) {
    int run = 0, arun = 0, urun = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      const int v = e < E ? cnt[e] : 0;
      const int np = (v + kUnitTokens - 1) / kUnitTokens;  // work units of <= 8 picks
      int inc = v, uinc = np;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, inc, off);
        const int uo = __shfl_up_sync(0xffffffffu, uinc, off);
        if (lane >= off) {
          inc += o;
          uinc += uo;
        }
      }
      const unsigned nz = __ballot_sync(0xffffffffu, v > 0);
      if (e < E) {
        cur[e] = run + inc - v;
        offsets[e] = run + inc - v;
        counts[e] = v;
        if (v > 0) act[arun + __popc(nz & ((1u << lane) - 1u))] = e;
        for (int i = 0; i < np; ++i) {
          UnitDesc& U = units[urun + uinc - np + i];
          U.e = e;
          U.M = min(kUnitTokens, v - i * kUnitTokens);
          U.pbase = run + inc - v + i * kUnitTokens;
          U.pad = 0;
        }
      }
      run += __shfl_sync(0xffffffffu, inc, 31);
      urun += __shfl_sync(0xffffffffu, uinc, 31);
      arun += __popc(nz);
    }
    if (lane == 0) {
      offsets[E] = run;
      *nact = arun;
      *nunits = urun;
      s_nunits = urun;
    }
  }
  __syncthreads();
  for (int r0 = 0; r0 < P; r0 += bd) {
    const int p = r0 + tid;
    int e = p < P ? __ldcg(idx + p) : -1;
    const bool valid = e >= 0 && e < E;
    if (!valid) e = -1;
    const unsigned same = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(same & ((1u << lane) - 1u));
    for (int wv = 0; wv < nwarps; ++wv) {
      if (warp == wv) {
        int base = 0;
        if (valid) base = cur[e];
        __syncwarp();
        if (valid) {
          perm[base + rank] = p;
          if (rank == 0) cur[e] = base + __popc(same);
        }
      }
      __syncthreads();
    }
  }
  // per-unit pick lists (perm was written by this block above)
  __threadfence_block();
  __syncthreads();
  for (int u = tid; u < s_nunits; u += bd) {
    UnitDesc& U = units[u];
    const int M = U.M, pb = U.pbase;
    for (int m = 0; m < kUnitTokens; ++m) {
      const int p = m < M ? __ldcg(perm + pb + m) : 0;
      const int t = p / k;
      U.pick[m] = m < M ? p : -1;
      U.tok[m] = m < M ? t : 0;
      U.xs[m] = m < M ? __ldcg(xscale + t) : 0.f;
      U.w[m] = m < M ? __ldcg(w + p) : 0.f;
    }
  }
}

namespace {

__global__ void __launch_bounds__(kRouterWarps * 32) router_kernel(RouterArgs a) {
  extern __shared__ float dsm[];
  __shared__ float red[kRouterWarps];
  __shared__ int last;
  logits_rows(a);
  convert_tokens(a, red);
  if (!a.fuse_select) return;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = (atomicAdd(&a.ws.sync[0], 1u) == gridDim.x - 1);
  __syncthreads();
  if (!last) return;
  __threadfence();
  const int warp = threadIdx.x >> 5;
  for (int t = warp; t < a.T; t += kRouterWarps)
    topk_warp(a.ws.logits + (size_t)t * a.E, a.bias, a.E, a.k, dsm + (size_t)warp * a.E, a.ws.idx + (size_t)t * a.k,
              a.ws.w + (size_t)t * a.k);
  __threadfence_block();
  __syncthreads();
  bucket_block(a.ws.idx, a.T * a.k, a.k, a.E, a.ws.counts, a.ws.offsets, a.ws.perm, a.ws.act, a.ws.nact,
               a.ws.units, a.ws.nunits, a.ws.w, a.ws.xscale, reinterpret_cast<int*>(dsm));
  if (threadIdx.x == 0) a.ws.sync[0] = 0u;
}

__global__ void __launch_bounds__(256) topk_kernel(const float* logits, const float* bias, int T, int E, int k,
                                                   int32_t* idx, float* w) {
  extern __shared__ float dsm[];
  const int warp = threadIdx.x >> 5;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  topk_warp(logits + (size_t)t * E, bias, E, k, dsm + (size_t)warp * E, idx + (size_t)t * k, w + (size_t)t * k);
}

__global__ void __launch_bounds__(1024) bucket_kernel(const int32_t* idx, int P, int k, int E, int32_t* counts,
                                                      int32_t* offsets, int32_t* perm, int32_t* act, int32_t* nact,
                                                      UnitDesc* units, int32_t* nunits, const float* w,
                                                      const float* xscale) {
  extern __shared__ int ism[];
  bucket_block(idx, P, k, E, counts, offsets, perm, act, nact, units, nunits, w, xscale, ism);
}

}  // namespace

cudaError_t launch_router(const RouterArgs& a, cudaStream_t s) {
  const size_t smem = (size_t)kRouterWarps * a.E * sizeof(float);
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(router_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    attr = true;
  }
  const int grid = (a.E + kRouterWarps - 1) / kRouterWarps;
  router_kernel<<<grid, kRouterWarps * 32, a.fuse_select ? smem : 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_topk(const float* logits, const float* bias, int T, int E, int k, int32_t* idx, float* w,
                        cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    attr = true;
  }
  topk_kernel<<<(T + 7) / 8, 256, (size_t)8 * E * sizeof(float), s>>>(logits, bias, T, E, k, idx, w);
  return cudaGetLastError();
}

cudaError_t launch_bucket(const int32_t* idx, int T, int k, int E, int32_t* counts, int32_t* offsets,
                          int32_t* perm, int32_t* act, int32_t* nact, UnitDesc* units, int32_t* nunits,
                          const float* w, const float* xscale, cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(bucket_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
    attr = true;
  }
  bucket_kernel<<<1, 1024, (size_t)2 * E * sizeof(int), s>>>(idx, T * k, k, E, counts, offsets, perm, act, nact,
                                                              units, nunits, w, xscale);
  return cudaGetLastError();
}

}  // namespace k3
