// decode_ffn.cu -- small-T expert FFN straight from the MXFP4 bytes (register decode).
//
// "kimi-k3-in-c deep dive", "four reductions", reduction 1: the experts stay MXFP4 and are
// multiplied on the nibbles, never expanded to a dense copy (value = E2M1[nibble] *
// 2^(scale-127), 32 values per scale).  On the GPU each expert's bytes are streamed from HBM
// exactly once per call, each lane's 16-byte chunk is turned into four f16x2 A fragments per
// word with the hardware e2m1x2 -> f16x2 conversion, and mma.m16n8k16 multiplies them with
// up to 8 routed tokens at a time (tokens are the n = 8 columns).  The E8M0 scale of a
// 32-column block is applied once per block: the block's two k16 steps accumulate into a
// zeroed fp32 fragment that is then added, times the scale, to the running fp32 sum.  Every
// product is exact (fp16 x fp16 into fp32) and all sums are fp32.
//
//   gateup_kernel: CTA = (routed expert, 32 rows of f); 8 warps split d; the partial sums
//                  are added in warp order, then h = silu(g) * u (SwiGLU) is stored as fp16
//                  B fragments with one power-of-two scale per (pick, 32 rows).
//   down_kernel:   CTA = (routed expert, 64 rows of d); 4 row groups x 2 halves of f; the
//                  outputs times the combine weight go to obuf[pick]; the last of a token's
//                  k picks to finish a 64-row chunk sums the k slots in slot order into y
//                  (fixed reduction order, independent of which CTA finishes last).
#include "k3moe_internal.cuh"

namespace k3 {
namespace {

__device__ __forceinline__ void dec4(uint32_t w, uint32_t (&a)[4]) {
  asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
      "mov.b32 {q0, q1, q2, q3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, q0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, q1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, q2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, q3;\n\t}"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
      : "r"(w));
}

__device__ __forceinline__ void mma_acc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_zero(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  const float z = 0.f;
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
}

// E8M0 byte -> 2^(s-127) as fp32 (s = 0 is the subnormal 2^-127).
__device__ __forceinline__ float e8m0f(uint32_t s) { return __uint_as_float(s ? (s << 23) : 0x00400000u); }

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint4 ld_stream16(const uint8_t* ptr, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr), "l"(pol));
  return v;
}

__device__ __forceinline__ uint2 ld_stream8(const uint8_t* ptr, uint64_t pol) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v2.u32 {%0,%1}, [%2], %3;"
               : "=r"(v.x), "=r"(v.y)
               : "l"(ptr), "l"(pol));
  return v;
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int s) {
  return s == 0 ? v.x : (s == 1 ? v.y : (s == 2 ? v.z : v.w));
}

__device__ __forceinline__ int fp16_scale_exp(float m) {
  if (!(m > 0.0f)) return 0;
  const int ex = (int)((__float_as_uint(m) >> 23) & 0xFFu) - 127;
  const int q = ex - 14;
  return q < -126 ? -126 : (q > 126 ? 126 : q);
}
__device__ __forceinline__ float exp2i(int q) { return __uint_as_float((uint32_t)(127 + q) << 23); }

constexpr int kWarps = 8;

// ------------------------------------------------------------------------ gate/up ---
__global__ void __launch_bounds__(kWarps * 32, 2) gateup_kernel(FfnArgs a) {
  __shared__ float red[kWarps][16][32];
  __shared__ __half hstage[8][32];
  __shared__ float s_hsc[8];
  __shared__ float s_xs[8];
  __shared__ int s_pick[8];

  const int chunks = a.f / 32;
  const int ai = blockIdx.x / chunks, c = blockIdx.x % chunks;
  if (ai >= *a.ws.nact) return;
  const int e = a.ws.act[ai];
  const int M = a.ws.counts[e], pbase = a.ws.offsets[e];
  const uint8_t* W = a.expert_ptr[e];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int ktiles = a.d / kTileCols;
  const int kt0 = warp * ktiles / kWarps, kt1 = (warp + 1) * ktiles / kWarps;
  const uint64_t pol = policy_evict_first();

  for (int n0 = 0; n0 < M; n0 += 8) {
    if (threadIdx.x < 8) {
      const int n = n0 + threadIdx.x;
      const int p = n < M ? a.ws.perm[pbase + n] : -1;
      s_pick[threadIdx.x] = p;
      s_xs[threadIdx.x] = p >= 0 ? a.ws.xscale[p / a.k] : 0.f;
    }
    const bool has = n0 + g < M;
    const int mypick = has ? a.ws.perm[pbase + n0 + g] : 0;
    const uint4* xb = reinterpret_cast<const uint4*>(a.ws.xfrag + (size_t)(mypick / a.k) * a.d) + t;

    float acc[2][2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[i][j][q] = 0.f;

    for (int kt = kt0; kt < kt1; ++kt) {
      uint4 nib[2][2][2];
      uint2 sc[2][2];
#pragma unroll
      for (int rg = 0; rg < 2; ++rg)
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const uint8_t* tp = W + ((size_t)((2 * c + rg) * ktiles + kt) * 2 + m) * kTileBytes;
          nib[rg][m][0] = ld_stream16(tp + lane * 16, pol);
          nib[rg][m][1] = ld_stream16(tp + 512 + lane * 16, pol);
          sc[rg][m] = ld_stream8(tp + kTileNibBytes + g * 8, pol);
        }
      uint4 xv[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) xv[b] = has ? __ldg(xb + (size_t)(4 * kt + b) * 4) : make_uint4(0, 0, 0, 0);

#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int u = b >> 1;
        float bacc[2][2][4];
#pragma unroll
        for (int st = 0; st < 2; ++st) {
          const int s = 2 * (b & 1) + st;
          const uint32_t b0 = st ? xv[b].z : xv[b].x, b1 = st ? xv[b].w : xv[b].y;
#pragma unroll
          for (int rg = 0; rg < 2; ++rg)
#pragma unroll
            for (int m = 0; m < 2; ++m) {
              uint32_t A[4];
              dec4(word_of(nib[rg][m][u], s), A);
              if (st == 0)
                mma_zero(bacc[rg][m], A, b0, b1);
              else
                mma_acc(bacc[rg][m], A, b0, b1);
            }
        }
#pragma unroll
        for (int rg = 0; rg < 2; ++rg)
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            const float s0 = e8m0f((sc[rg][m].x >> (8 * b)) & 0xFFu);
            const float s8 = e8m0f((sc[rg][m].y >> (8 * b)) & 0xFFu);
            acc[rg][m][0] = fmaf(bacc[rg][m][0], s0, acc[rg][m][0]);
            acc[rg][m][1] = fmaf(bacc[rg][m][1], s0, acc[rg][m][1]);
            acc[rg][m][2] = fmaf(bacc[rg][m][2], s8, acc[rg][m][2]);
            acc[rg][m][3] = fmaf(bacc[rg][m][3], s8, acc[rg][m][3]);
          }
      }
    }

#pragma unroll
    for (int rg = 0; rg < 2; ++rg)
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int q = 0; q < 4; ++q) red[warp][(rg * 2 + m) * 4 + q][lane] = acc[rg][m][q];
    __syncthreads();

    if (warp == 0) {
      float hv[2][4];
      float mx0 = 0.f, mx1 = 0.f;
#pragma unroll
      for (int rg = 0; rg < 2; ++rg)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float gs = 0.f, us = 0.f;
          for (int w = 0; w < kWarps; ++w) {
            gs += red[w][(rg * 2 + 0) * 4 + q][lane];
            us += red[w][(rg * 2 + 1) * 4 + q][lane];
          }
          const float xs = s_xs[2 * t + (q & 1)];
          const float gt = gs * xs, ut = us * xs;
          const float h = gt / (1.0f + expf(-gt)) * ut;
          hv[rg][q] = h;
          if (q & 1)
            mx1 = fmaxf(mx1, fabsf(h));
          else
            mx0 = fmaxf(mx0, fabsf(h));
        }
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      const int q0 = fp16_scale_exp(mx0), q1 = fp16_scale_exp(mx1);
      const float i0 = exp2i(-q0), i1 = exp2i(-q1);
#pragma unroll
      for (int rg = 0; rg < 2; ++rg)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int r = 16 * rg + g + 8 * (q >> 1);
          const int n = 2 * t + (q & 1);
          hstage[n][r] = __float2half_rn(hv[rg][q] * ((q & 1) ? i1 : i0));
        }
      if (g == 0) {
        s_hsc[2 * t] = exp2i(q0);
        s_hsc[2 * t + 1] = exp2i(q1);
      }
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      const int n = threadIdx.x >> 2, tq = threadIdx.x & 3;
      const int p = s_pick[n];
      if (p >= 0) {
        __align__(16) __half hh[8];
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          hh[4 * s + 0] = hstage[n][16 * s + 2 * tq];
          hh[4 * s + 1] = hstage[n][16 * s + 2 * tq + 1];
          hh[4 * s + 2] = hstage[n][16 * s + 2 * tq + 8];
          hh[4 * s + 3] = hstage[n][16 * s + 2 * tq + 9];
        }
        *reinterpret_cast<uint4*>(a.ws.hfrag + (size_t)p * a.f + (size_t)(c * 4 + tq) * 8) =
            *reinterpret_cast<const uint4*>(hh);
        if (tq == 0) a.ws.hscale[(size_t)p * chunks + c] = s_hsc[n];
      }
    }
    __syncthreads();
  }
}

// --------------------------------------------------------------------- down+combine ---
__global__ void __launch_bounds__(kWarps * 32, 2) down_kernel(FfnArgs a) {
  __shared__ float red[4][4][32];
  __shared__ int s_pick[8];
  __shared__ float s_w[8];
  __shared__ int s_last[8];

  const int chunks = a.d / 64;
  const int ai = blockIdx.x / chunks, c = blockIdx.x % chunks;
  if (ai >= *a.ws.nact) return;
  const int e = a.ws.act[ai];
  const int M = a.ws.counts[e], pbase = a.ws.offsets[e];
  const uint8_t* W = a.expert_ptr[e] + gateup_region_bytes(a.d, a.f);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int rgl = warp & 3, half = warp >> 2;
  const int rg = 4 * c + rgl;
  const int ktiles = a.f / kTileCols;
  const int nblk = a.f / 32;
  int kt0, kt1;
  if (ktiles >= 2) {
    kt0 = half * ktiles / 2;
    kt1 = (half + 1) * ktiles / 2;
  } else {
    kt0 = 0;
    kt1 = half == 0 ? ktiles : 0;
  }
  const uint64_t pol = policy_evict_first();

  for (int n0 = 0; n0 < M; n0 += 8) {
    if (threadIdx.x < 8) {
      const int n = n0 + threadIdx.x;
      const int p = n < M ? a.ws.perm[pbase + n] : -1;
      s_pick[threadIdx.x] = p;
      s_w[threadIdx.x] = p >= 0 ? a.ws.w[p] : 0.f;
    }
    __syncthreads();
    const bool has = n0 + g < M;
    const int mypick = has ? s_pick[g] : 0;
    const uint4* hb = reinterpret_cast<const uint4*>(a.ws.hfrag + (size_t)mypick * a.f) + t;
    const int p0 = s_pick[2 * t], p1 = s_pick[2 * t + 1];
    const float* hs0 = a.ws.hscale + (size_t)(p0 >= 0 ? p0 : 0) * nblk;
    const float* hs1 = a.ws.hscale + (size_t)(p1 >= 0 ? p1 : 0) * nblk;

    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int kt = kt0; kt < kt1; ++kt) {
      const uint8_t* tp = W + ((size_t)rg * ktiles + kt) * kTileBytes;
      const uint4 n_0 = ld_stream16(tp + lane * 16, pol);
      const uint4 n_1 = ld_stream16(tp + 512 + lane * 16, pol);
      const uint2 sc = ld_stream8(tp + kTileNibBytes + g * 8, pol);
      uint4 hv[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) hv[b] = has ? __ldg(hb + (size_t)(4 * kt + b) * 4) : make_uint4(0, 0, 0, 0);
      float h0[4], h1[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        h0[b] = p0 >= 0 ? __ldg(hs0 + 4 * kt + b) : 0.f;
        h1[b] = p1 >= 0 ? __ldg(hs1 + 4 * kt + b) : 0.f;
      }
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint4& nv = (b >> 1) ? n_1 : n_0;
        float bacc[4];
#pragma unroll
        for (int st = 0; st < 2; ++st) {
          const int s = 2 * (b & 1) + st;
          uint32_t A[4];
          dec4(word_of(nv, s), A);
          const uint32_t b0 = st ? hv[b].z : hv[b].x, b1 = st ? hv[b].w : hv[b].y;
          if (st == 0)
            mma_zero(bacc, A, b0, b1);
          else
            mma_acc(bacc, A, b0, b1);
        }
        const float s0 = e8m0f((sc.x >> (8 * b)) & 0xFFu);
        const float s8 = e8m0f((sc.y >> (8 * b)) & 0xFFu);
        acc[0] = fmaf(bacc[0], s0 * h0[b], acc[0]);
        acc[1] = fmaf(bacc[1], s0 * h1[b], acc[1]);
        acc[2] = fmaf(bacc[2], s8 * h0[b], acc[2]);
        acc[3] = fmaf(bacc[3], s8 * h1[b], acc[3]);
      }
    }
    if (half == 1) {
#pragma unroll
      for (int q = 0; q < 4; ++q) red[rgl][q][lane] = acc[q];
    }
    __syncthreads();
    if (half == 0) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float o = acc[q] + red[rgl][q][lane];
        const int n = 2 * t + (q & 1);
        const int p = s_pick[n];
        if (p >= 0) {
          const int row = 64 * c + 16 * rgl + g + 8 * (q >> 1);
          a.ws.obuf[(size_t)p * a.d + row] = o * s_w[n];
        }
      }
      __threadfence();
    }
    __syncthreads();
    if (threadIdx.x < 8) {
      const int p = s_pick[threadIdx.x];
      int last = 0;
      if (p >= 0) {
        const int tok = p / a.k;
        last = atomicAdd(&a.ws.arrive[(size_t)tok * chunks + c], 1) == a.k - 1;
      }
      s_last[threadIdx.x] = last;
    }
    __syncthreads();
    for (int n = 0; n < 8; ++n) {
      if (!s_last[n]) continue;
      __threadfence();
      const int tok = s_pick[n] / a.k;
      if (threadIdx.x < 64) {
        const int row = 64 * c + threadIdx.x;
        float y = 0.f;
        for (int slot = 0; slot < a.k; ++slot) y += __ldcg(a.ws.obuf + ((size_t)tok * a.k + slot) * a.d + row);
        a.y[(size_t)tok * a.d + row] = y;
      }
      if (threadIdx.x == 0) a.ws.arrive[(size_t)tok * chunks + c] = 0;
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_gateup(const FfnArgs& a, cudaStream_t s) {
  gateup_kernel<<<a.max_tasks * (a.f / 32), kWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_down(const FfnArgs& a, cudaStream_t s) {
  down_kernel<<<a.max_tasks * (a.d / 64), kWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace k3
