// router.cu -- router logits, sigmoid + bias top-k selection, and token-to-expert bucketing.
//
// Routing rule ("kimi-k3-in-c deep dive": "what you learn", router paragraph, and the
// invariants table, row 5): sigmoid scores; the bias steers the selection only; the picked
// experts are mixed with weights from the unbiased scores, renormalised to sum 1.  The pages
// pick 16 of 896 experts (glossary entry MoE).
//
// GPU design: the router is a GEMV over W_r (fp32, [E][d]) with two warps per expert row (one
// per half of d, 14 loads in flight per lane) and the tokens staged in shared memory 4 at a time,
// so W_r is read once per call.  The same pass converts each token to fp16 fragments.  For
// small T the last CTA to finish (atomic ticket) also runs the top-k and the bucketing, which
// saves two launches on the single-token path.  Top-k is a warp per token: k rounds of a
// warp-wide (key desc, id asc) argmax over the keys kept in shared memory.  Bucketing is
// deterministic: counts by shared-memory atomics (order-free), an exclusive scan, and a
// stable scatter in rounds where __match_any_sync ranks equal experts inside a warp and the
// warps of a round take their turn in order.
#include <algorithm>

#include "k3moe_internal.cuh"

namespace k3 {
namespace {

constexpr int kRouterWarps = 8;  // 2 warps per expert row (each half of d)
constexpr int kWarpsPerRow = 2;
constexpr int kRowsPerCta = kRouterWarps / kWarpsPerRow;
constexpr int kTokTile = 4;      // tokens staged in shared memory at a time

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

// Stage tokens [t0, t0+nt) of x (bf16) into shared memory with 16-byte loads.
__device__ void stage_tokens(const RouterArgs& a, int t0, int nt, uint16_t* xs) {
  const int n16 = nt * a.d / 8;
  const uint4* src = reinterpret_cast<const uint4*>(a.x + (size_t)t0 * a.d);
  uint4* dst = reinterpret_cast<uint4*>(xs);
  for (int i = threadIdx.x; i < n16; i += blockDim.x) dst[i] = __ldg(src + i);
}

// x row (bf16, in shared memory) -> fp16 B-fragment row with a per-token power-of-two scale.
__device__ void convert_token(const RouterArgs& a, int t, const uint16_t* xr, float* red) {
  float m = 0.f;
  for (int j = threadIdx.x * 2; j < a.d; j += blockDim.x * 2) {
    const uint32_t v = *reinterpret_cast<const uint32_t*>(xr + j);
    m = fmaxf(m, fmaxf(fabsf(bf16_lo(v)), fabsf(bf16_hi(v))));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  m = red[0];
  for (int i = 1; i < (int)(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
  const int q = fp16_scale_exp(m);
  const float inv = exp2i(-q);
  const int items = (a.d / 32) * 4;
  for (int it = threadIdx.x; it < items; it += blockDim.x) {
    const int blk = it >> 2, tq = it & 3;
    __align__(16) __half h[8];
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int kb = 32 * blk + 16 * s + 2 * tq;
      const uint32_t p0 = *reinterpret_cast<const uint32_t*>(xr + kb);
      const uint32_t p1 = *reinterpret_cast<const uint32_t*>(xr + kb + 8);
      h[4 * s + 0] = __float2half_rn(bf16_lo(p0) * inv);
      h[4 * s + 1] = __float2half_rn(bf16_hi(p0) * inv);
      h[4 * s + 2] = __float2half_rn(bf16_lo(p1) * inv);
      h[4 * s + 3] = __float2half_rn(bf16_hi(p1) * inv);
    }
    *reinterpret_cast<uint4*>(a.ws.xfrag + (size_t)t * a.d + (size_t)it * 8) = *reinterpret_cast<uint4*>(h);
  }
  if (threadIdx.x == 0) a.ws.xscale[t] = exp2i(q);
  __syncthreads();
}

// --------------------------------------------------------------------------- logits ---
// CTA = kRowsPerCta expert rows; warp w handles row w / kWarpsPerRow, part w % kWarpsPerRow of
// d; the partial sums are added in a fixed order.  Tokens are staged kTokTile at a time; the CTA
// with blockIdx == t % grid also converts token t to fp16 fragments.
__device__ void logits_and_convert(const RouterArgs& a, uint16_t* xs, float* red, float* part) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * kRowsPerCta + warp / kWarpsPerRow;
  const int qt = warp % kWarpsPerRow;
  const int nq = a.d / 4, span = nq / kWarpsPerRow, q0 = qt * span, q1 = q0 + span;
  const float4* wr = reinterpret_cast<const float4*>(a.Wr + (size_t)(e < a.E ? e : 0) * a.d);
  constexpr int kB = 14;  // W_r loads in flight per lane
  pdl_entry();
  for (int t0 = 0; t0 < a.T; t0 += kTokTile) {
    const int nt = min(kTokTile, a.T - t0);
    __syncthreads();
    stage_tokens(a, t0, nt, xs);
    __syncthreads();
    for (int tt = 0; tt < nt; ++tt)
      if ((t0 + tt) % (int)gridDim.x == (int)blockIdx.x) convert_token(a, t0 + tt, xs + (size_t)tt * a.d, red);
    float acc[kTokTile] = {0.f, 0.f, 0.f, 0.f};
    if (e < a.E) {
      for (int qb = q0 + lane; qb < q1; qb += 32 * kB) {
        float4 wv[kB];
#pragma unroll
        for (int j = 0; j < kB; ++j) {
          const int q = qb + 32 * j;
          wv[j] = q < q1 ? __ldg(wr + q) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < kB; ++j) {
          const int q = qb + 32 * j;
          if (q < q1) {
#pragma unroll
            for (int tt = 0; tt < kTokTile; ++tt) {
              if (tt < nt) {
                const uint2 xv = *reinterpret_cast<const uint2*>(xs + (size_t)tt * a.d + 4 * q);
                acc[tt] = fmaf(bf16_lo(xv.x), wv[j].x, acc[tt]);
                acc[tt] = fmaf(bf16_hi(xv.x), wv[j].y, acc[tt]);
                acc[tt] = fmaf(bf16_lo(xv.y), wv[j].z, acc[tt]);
                acc[tt] = fmaf(bf16_hi(xv.y), wv[j].w, acc[tt]);
              }
            }
          }
        }
      }
    }
#pragma unroll
    for (int tt = 0; tt < kTokTile; ++tt) {
      float v = acc[tt];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0) part[warp * kTokTile + tt] = v;
    }
    __syncthreads();
    if (qt == 0 && lane < nt && e < a.E) {
      const float* pp = part + warp * kTokTile + lane;
      float v = pp[0];
#pragma unroll
      for (int h = 1; h < kWarpsPerRow; ++h) v += pp[h * kTokTile];
      a.ws.logits[(size_t)(t0 + lane) * a.E + e] = v;
    }
  }
}

}  // namespace

// ---------------------------------------------------------------------------- top-k ---
// Key as an unsigned integer with the same order as the float (larger key -> larger integer).
__device__ __forceinline__ uint32_t ord_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// a is ranked before b: larger key, or equal key and lower expert id
__device__ __forceinline__ bool ranks_before(uint32_t ua, int ia, uint32_t ub, int ib) {
  return ua > ub || (ua == ub && ia < ib);
}

// Bitonic sort of the warp's 32*R (key, id) pairs into rank order (best first); element
// i = 32*j + lane lives in register j of lane `lane`.
template <int R>
__device__ __forceinline__ void warp_sort(uint32_t (&u)[R], int (&id)[R]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 32 * R; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride >= 32) {
        const int js = stride / 32;
#pragma unroll
        for (int j = 0; j < R; ++j) {
          const int jp = j ^ js;
          if (j < jp) {
            const bool asc = (((32 * j + lane) & size) == 0);  // block ordered best-first
            const bool swap = asc ? ranks_before(u[jp], id[jp], u[j], id[j]) : ranks_before(u[j], id[j], u[jp], id[jp]);
            if (swap) {
              const uint32_t tu = u[j];
              const int ti = id[j];
              u[j] = u[jp];
              id[j] = id[jp];
              u[jp] = tu;
              id[jp] = ti;
            }
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < R; ++j) {
          const uint32_t ou = __shfl_xor_sync(0xffffffffu, u[j], stride);
          const int oi = __shfl_xor_sync(0xffffffffu, id[j], stride);
          const int i = 32 * j + lane;
          const bool keep_first = (((i & size) == 0) == ((i & stride) == 0));
          if (keep_first != ranks_before(u[j], id[j], ou, oi)) {
            u[j] = ou;
            id[j] = oi;
          }
        }
      }
    }
  }
}

// Merge a ranked 32-list held one per lane (a) with another (b) into the ranked best 32 of both.
__device__ __forceinline__ void warp_merge32(uint32_t& au, int& ai, uint32_t bu, int bi) {
  const int lane = threadIdx.x & 31;
  // a ascending by rank, b reversed: the elementwise better of the two is a bitonic sequence
  // holding the best 32 of the union
  const uint32_t ru = __shfl_sync(0xffffffffu, bu, 31 - lane);
  const int ri = __shfl_sync(0xffffffffu, bi, 31 - lane);
  if (ranks_before(ru, ri, au, ai)) {
    au = ru;
    ai = ri;
  }
#pragma unroll
  for (int stride = 16; stride > 0; stride >>= 1) {
    const uint32_t ou = __shfl_xor_sync(0xffffffffu, au, stride);
    const int oi = __shfl_xor_sync(0xffffffffu, ai, stride);
    const bool keep_first = (lane & stride) == 0;
    if (keep_first != ranks_before(au, ai, ou, oi)) {
      au = ou;
      ai = oi;
    }
  }
}

constexpr int kTopkThreads = 256;
constexpr int kSortR = 4;  // per-warp sort chunk: 32 * kSortR keys

// The whole block selects the k largest keys (k <= 32) of one token.  Shared memory: ku/sg =
// E words each (ordered keys, unbiased sigmoid scores), cand = 8 * 32 (key, id) pairs.  Each
// thread scores E/256 experts; each warp sorts its slice in chunks of 128 and keeps a ranked
// top-32; the 8 lists are merged by warp 0.  The picks go to idx_out/w_out (global) and, when
// given, to the shared-memory copies idx_s/w_s.
__device__ void topk_block(const float* logits_row, const float* bias, int E, int k, uint32_t* ku, float* sg,
                           uint2* cand, int32_t* idx_out, float* w_out, int32_t* idx_s = nullptr,
                           float* w_s = nullptr) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nw = blockDim.x >> 5;
  // scores: every thread issues all of its loads before using any of them
  constexpr int kB = 8;
  for (int e0 = 0; e0 < E; e0 += (int)blockDim.x * kB) {
    float z[kB], b[kB];
#pragma unroll
    for (int j = 0; j < kB; ++j) {
      const int e = e0 + (int)blockDim.x * j + tid;
      z[j] = e < E ? __ldcg(logits_row + e) : 0.f;
      b[j] = (bias && e < E) ? __ldg(bias + e) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kB; ++j) {
      const int e = e0 + (int)blockDim.x * j + tid;
      if (e < E) {
        const float s = sigmoidf_acc(z[j]);
        sg[e] = s;
        ku[e] = ord_key(s + b[j]);
      }
    }
  }
  __syncthreads();
  // per-warp ranked top-32 of its slice
  const int per = (E + nw - 1) / nw;
  const int ea = min(E, warp * per), eb = min(E, ea + per);
  uint32_t bu = 0u;
  int bi = 0x7fffffff;
  for (int c0 = ea; c0 < eb; c0 += 32 * kSortR) {
    uint32_t u[kSortR];
    int id[kSortR];
#pragma unroll
    for (int j = 0; j < kSortR; ++j) {
      const int e = c0 + 32 * j + lane;
      const bool in = e < eb;
      u[j] = in ? ku[e] : 0u;
      id[j] = in ? e : 0x7fffffff;
    }
    warp_sort<kSortR>(u, id);
    warp_merge32(bu, bi, u[0], id[0]);
  }
  // pairwise tree of merges: at level h, warp w (w % 2h == 0) merges warp w + h's list into its own
  cand[warp * 32 + lane] = make_uint2(bu, (uint32_t)bi);
  for (int h = 1; h < nw; h <<= 1) {
    __syncthreads();
    if (warp % (2 * h) == 0 && warp + h < nw) {
      const uint2 c = cand[(warp + h) * 32 + lane];
      warp_merge32(bu, bi, c.x, (int)c.y);
      cand[warp * 32 + lane] = make_uint2(bu, (uint32_t)bi);
    }
  }
  if (warp == 0) {
    const int ai = bi;
    const float s = lane < k ? sg[ai] : 0.f;
    float tot = s;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
    if (lane < k) {
      const float wv = s / tot;
      idx_out[lane] = ai;
      w_out[lane] = wv;
      if (idx_s) {
        idx_s[lane] = ai;
        w_s[lane] = wv;
      }
    }
  }
  __syncthreads();
}

// ------------------------------------------------------------------------ bucketing ---
// Whole-block deterministic bucketing of P picks.  smem: 2*E ints, plus P ints when
// perm_smem (small P: the unit descriptors then read perm from shared memory).
// whist: smem also holds [nwarps][E] per-warp expert counts (zero on entry and on exit), which
// replaces the warp-by-warp stable scatter with three barriers per block of picks.
__device__ void bucket_block(const int32_t* idx, int P, int k, int E, int32_t* counts, int32_t* offsets,
                             int32_t* perm, int32_t* act, int32_t* nact, UnitDesc* units, int32_t* nunits,
                             const float* w, const float* xscale, int* smem, bool perm_smem, bool iw_smem = false,
                             int* whist = nullptr, bool fill_units = true) {
  // iw_smem: idx and w are shared-memory arrays of this block (else global, written earlier)
  auto ld_idx = [&](int p) { return iw_smem ? idx[p] : __ldcg(idx + p); };
  auto ld_w = [&](int p) { return iw_smem ? w[p] : __ldcg(w + p); };
  __shared__ int s_nunits;
  int* cnt = smem;
  int* cur = smem + E;
  int* sperm = smem + 2 * E;
  const int tid = threadIdx.x, bd = blockDim.x, warp = tid >> 5, lane = tid & 31, nwarps = bd >> 5;
  for (int e = tid; e < E; e += bd) cnt[e] = 0;
  __syncthreads();
  for (int p0 = 0; p0 < P; p0 += bd * 8) {  // 8 loads in flight per thread
    int ev[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int p = p0 + j * bd + tid;
      ev[j] = p < P ? ld_idx(p) : -1;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {  // one shared-memory atomic per distinct expert of the warp
      const int e = (ev[j] >= 0 && ev[j] < E) ? ev[j] : -1;
      const unsigned same = __match_any_sync(0xffffffffu, e);
      if (e >= 0 && (same & ((1u << lane) - 1u)) == 0u) atomicAdd(&cnt[e], __popc(same));
    }
  }
  __syncthreads();
  // block-wide exclusive scan over experts of (picks, active flag, work units); each thread owns
  // a contiguous range of experts, so every output stays in expert-id order
  __shared__ int wsum[3][32];
  const int per = (E + bd - 1) / bd;
  const int ea = min(E, tid * per), eb = min(E, ea + per);
  int cs = 0, as = 0, us = 0;
  for (int e = ea; e < eb; ++e) {
    const int v = cnt[e];
    cs += v;
    as += v > 0;
    us += (v + kUnitTokens - 1) / kUnitTokens;
  }
  int ci = cs, ai = as, ui = us;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int c2 = __shfl_up_sync(0xffffffffu, ci, off), a2 = __shfl_up_sync(0xffffffffu, ai, off),
              u2 = __shfl_up_sync(0xffffffffu, ui, off);
    if (lane >= off) {
      ci += c2;
      ai += a2;
      ui += u2;
    }
  }
  if (lane == 31) {
    wsum[0][warp] = ci;
    wsum[1][warp] = ai;
    wsum[2][warp] = ui;
  }
  __syncthreads();
  if (warp == 0) {
    int c0 = lane < nwarps ? wsum[0][lane] : 0, a0 = lane < nwarps ? wsum[1][lane] : 0,
        u0 = lane < nwarps ? wsum[2][lane] : 0;
    int cc = c0, aa = a0, uu = u0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int c2 = __shfl_up_sync(0xffffffffu, cc, off), a2 = __shfl_up_sync(0xffffffffu, aa, off),
                u2 = __shfl_up_sync(0xffffffffu, uu, off);
      if (lane >= off) {
        cc += c2;
        aa += a2;
        uu += u2;
      }
    }
    __syncwarp();
    if (lane < nwarps) {
      wsum[0][lane] = cc - c0;
      wsum[1][lane] = aa - a0;
      wsum[2][lane] = uu - u0;
    }
    if (lane == 31) {
      offsets[E] = cc;
      *nact = aa;
      *nunits = uu;
      s_nunits = uu;
    }
  }
  __syncthreads();
  {
    int run = wsum[0][warp] + ci - cs, arun = wsum[1][warp] + ai - as, urun = wsum[2][warp] + ui - us;
    for (int e = ea; e < eb; ++e) {
      const int v = cnt[e];
      cur[e] = run;
      offsets[e] = run;
      counts[e] = v;
      if (v > 0) act[arun++] = e;
      const int np = (v + kUnitTokens - 1) / kUnitTokens;
      for (int i = 0; i < (fill_units ? np : 0); ++i) {
        UnitDesc& U = units[urun + i];
        U.e = e;
        U.M = min(kUnitTokens, v - i * kUnitTokens);
        U.pbase = run + i * kUnitTokens;
        U.pad = 0;
      }
      urun += np;
      run += v;
    }
  }
  __syncthreads();
  for (int r0 = 0; r0 < P && whist; r0 += bd) {
    // stable position = running offset of the expert + picks of it in earlier warps of this
    // block + rank inside the warp
    const int p = r0 + tid;
    int e = p < P ? ld_idx(p) : -1;
    const bool valid = e >= 0 && e < E;
    if (!valid) e = -1;
    const unsigned same = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(same & ((1u << lane) - 1u));
    if (valid && rank == 0) whist[warp * E + e] = __popc(same);
    __syncthreads();
    if (valid) {
      int base = cur[e];
      for (int w2 = 0; w2 < warp; ++w2) base += whist[w2 * E + e];
      perm[base + rank] = p;
      if (perm_smem) sperm[base + rank] = p;
    }
    __syncthreads();
    if (valid && rank == 0) {
      atomicAdd(&cur[e], __popc(same));
      whist[warp * E + e] = 0;
    }
    __syncthreads();
  }
  for (int r0 = 0; r0 < P && !whist; r0 += bd) {
    const int p = r0 + tid;
    int e = p < P ? ld_idx(p) : -1;
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
          if (perm_smem) sperm[base + rank] = p;
          if (rank == 0) cur[e] = base + __popc(same);
        }
      }
      __syncthreads();
    }
  }
  // per-unit pick lists: one thread per (unit, slot m); only the register-decode FFN reads them
  if (!fill_units) return;
  __threadfence_block();
  __syncthreads();
  const int nu = s_nunits;
  for (int um = tid; um < nu * kUnitTokens; um += bd) {
    const int u = um / kUnitTokens, m = um % kUnitTokens;
    UnitDesc& U = units[u];
    const int M = __ldcg(&U.M), pb = __ldcg(&U.pbase);
    const int p = m < M ? (perm_smem ? sperm[pb + m] : __ldcg(perm + pb + m)) : 0;
    const int t = p / k;
    U.pick[m] = m < M ? p : -1;
    U.tok[m] = m < M ? t : 0;
    U.xs[m] = m < M ? __ldcg(xscale + t) : 0.f;
    U.w[m] = m < M ? ld_w(p) : 0.f;
  }
}

// Bucketing of a few picks (P <= blockDim, at most kUnitTokens picks per expert), all in
// shared memory: the same counts, offsets, stable perm, active list and work units as
// bucket_block.  The rank of pick p is the number of picks with a lower expert id, or the same
// expert and a lower pick id; each run of equal experts in rank order is one unit.
__device__ void bucket_small(const int32_t* sidx, const float* sw, int P, int k, int E, int32_t* counts,
                             int32_t* offsets, int32_t* perm, int32_t* act, int32_t* nact, UnitDesc* units,
                             int32_t* nunits, const float* xscale, int* smem) {
  int* sperm = smem;      // [P] pick at rank r
  int* sel = smem + P;    // [P] expert at rank r
  const int tid = threadIdx.x;
  if (tid < P) {
    const int e = sidx[tid];
    int r = 0;
    for (int q = 0; q < P; ++q) {
      const int eq = sidx[q];
      r += (eq < e) || (eq == e && q < tid);
    }
    sperm[r] = tid;
    sel[r] = e;
  }
  __syncthreads();
  const bool start = tid < P && (tid == 0 || sel[tid - 1] != sel[tid]);
  const int nd = __syncthreads_count(start);
  if (tid < P) {
    perm[tid] = sperm[tid];
    if (start) {
      int g = 0;
      for (int q = 1; q <= tid; ++q) g += sel[q - 1] != sel[q];
      int M = 1;
      while (tid + M < P && sel[tid + M] == sel[tid]) ++M;
      act[g] = sel[tid];
      UnitDesc& U = units[g];
      U.e = sel[tid];
      U.M = M;
      U.pbase = tid;
      U.pad = 0;
#pragma unroll
      for (int m = 0; m < kUnitTokens; ++m) {
        const int pk = m < M ? sperm[tid + m] : -1;
        const int t = m < M ? pk / k : 0;
        U.pick[m] = pk;
        U.tok[m] = t;
        U.xs[m] = m < M ? xscale[t] : 0.f;  // shared-memory copy (T <= kUnitTokens)
        U.w[m] = m < M ? sw[pk] : 0.f;
      }
    }
  }
  for (int e = tid; e < E; e += blockDim.x) {
    int lo = 0, hi = P;  // first rank with expert >= e
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (sel[mid] < e) lo = mid + 1; else hi = mid;
    }
    int lo2 = lo, hi2 = P;  // first rank with expert > e
    while (lo2 < hi2) {
      const int mid = (lo2 + hi2) >> 1;
      if (sel[mid] <= e) lo2 = mid + 1; else hi2 = mid;
    }
    offsets[e] = lo;
    counts[e] = lo2 - lo;
  }
  if (tid == 0) {
    offsets[E] = P;
    *nact = nd;
    *nunits = nd;
  }
}

// Bucketing of at most 32 picks (T <= kUnitTokens) by one warp: the same stable perm, active
// list and work units as bucket_small, without the per-expert counts and offsets.  Lane q holds
// pick q; its rank is the number of picks with a lower expert id, or the same expert and a lower
// pick id.  A unit starts at each rank whose expert differs from the previous rank's.
// smem: 2 * 32 ints.  Called by the whole of warp 0.
__device__ void bucket_warp(const int32_t* sidx, const float* sw, int P, int k, int32_t* perm, int32_t* act,
                            int32_t* nact, UnitDesc* units, int32_t* nunits, const float* xscale, int* smem) {
  int* sel = smem;         // [32] expert at rank r
  int* sperm = smem + 32;  // [32] pick at rank r
  const int lane = threadIdx.x & 31;
  const int e = lane < P ? sidx[lane] : 0x7fffffff;
  int r = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int ej = __shfl_sync(0xffffffffu, e, j);
    r += (ej < e) || (ej == e && j < lane);
  }
  if (lane < P) {
    sel[r] = e;
    sperm[r] = lane;
  }
  __syncwarp();
  const int my = lane < P ? sel[lane] : -1;
  const int prev = __shfl_up_sync(0xffffffffu, my, 1);
  const bool start = lane < P && (lane == 0 || prev != my);
  const unsigned b = __ballot_sync(0xffffffffu, start);
  if (lane < P) perm[lane] = sperm[lane];
  if (start) {
    const int g = __popc(b & ((1u << lane) - 1u));
    const unsigned after = lane == 31 ? 0u : (b >> (lane + 1));
    const int M = after ? __ffs(after) : P - lane;  // ranks up to the next start
    act[g] = my;
    int pk[kUnitTokens], tk[kUnitTokens];
    float xv[kUnitTokens], wv[kUnitTokens];
#pragma unroll
    for (int m = 0; m < kUnitTokens; ++m) {
      pk[m] = m < M ? sperm[lane + m] : -1;
      tk[m] = m < M ? pk[m] / k : 0;
      xv[m] = m < M ? xscale[tk[m]] : 0.f;
      wv[m] = m < M ? sw[pk[m]] : 0.f;
    }
    int4* U = reinterpret_cast<int4*>(units + g);  // 9 x 16 bytes: header, pick, tok, xs, w
    U[0] = make_int4(my, M, lane, 0);
    U[1] = make_int4(pk[0], pk[1], pk[2], pk[3]);
    U[2] = make_int4(pk[4], pk[5], pk[6], pk[7]);
    U[3] = make_int4(tk[0], tk[1], tk[2], tk[3]);
    U[4] = make_int4(tk[4], tk[5], tk[6], tk[7]);
    float4* Uf = reinterpret_cast<float4*>(U);
    Uf[5] = make_float4(xv[0], xv[1], xv[2], xv[3]);
    Uf[6] = make_float4(xv[4], xv[5], xv[6], xv[7]);
    Uf[7] = make_float4(wv[0], wv[1], wv[2], wv[3]);
    Uf[8] = make_float4(wv[4], wv[5], wv[6], wv[7]);
  }
  if (lane == 0) {
    *nact = __popc(b);
    *nunits = __popc(b);
  }
}

// counts[e] and offsets[e] (e < E) of picks already in rank order (sel, P entries), whole block
__device__ void counts_from_sorted(const int* sel, int P, int E, int32_t* counts, int32_t* offsets) {
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int lo = 0, hi = P;  // first rank with expert >= e
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (sel[mid] < e) lo = mid + 1; else hi = mid;
    }
    int lo2 = lo, hi2 = P;  // first rank with expert > e
    while (lo2 < hi2) {
      const int mid = (lo2 + hi2) >> 1;
      if (sel[mid] <= e) lo2 = mid + 1; else hi2 = mid;
    }
    offsets[e] = lo;
    counts[e] = lo2 - lo;
  }
  if (threadIdx.x == 0) offsets[E] = P;
}

namespace {

__host__ inline size_t fused_select_smem(int E, int P) {
  return (size_t)(2 * E + 2) * 4 + 256 * 8 + ((size_t)2 * P + std::max<size_t>(2 * (size_t)E + P, 64)) * 4;
}

__global__ void __launch_bounds__(kRouterWarps * 32) router_kernel(RouterArgs a) {
  extern __shared__ __align__(16) uint8_t rsm[];
  __shared__ float red[kRouterWarps];
  __shared__ float part[kRouterWarps * kTokTile];
  __shared__ int last;
  logits_and_convert(a, reinterpret_cast<uint16_t*>(rsm), red, part);  // (waits on the grid dependency)
  if (!a.fuse_select) return;
  // last-block election: the barrier orders the CTA's logit and fragment writes before thread 0's
  // release; the last CTA's acquire (then its barrier) makes every CTA's writes visible to it
  __syncthreads();
  if (threadIdx.x == 0) last = (atom_add_acq_rel(&a.ws.sync[0], 1u) == gridDim.x - 1);
  __syncthreads();
  if (!last) return;
  // shared memory of the last block: [ku: E][sg: E][cand: 256 x 8 bytes][idx: P][w: P][bucketing: 2E + P]
  const int P = a.T * a.k;
  uint32_t* ku = reinterpret_cast<uint32_t*>(rsm);
  float* sg = reinterpret_cast<float*>(ku + a.E);
  uint2* cand = reinterpret_cast<uint2*>(sg + a.E);  // word offset 2E: 8-byte aligned
  int32_t* sidx = reinterpret_cast<int32_t*>(cand + 256);
  float* sw = reinterpret_cast<float*>(sidx + P);
  int* bsm = reinterpret_cast<int*>(sw + P);
  // token scales for the work units, loaded now so that the top-k hides their latency
  __shared__ float sxs[kUnitTokens];
  if (threadIdx.x < min(a.T, kUnitTokens)) sxs[threadIdx.x] = __ldcg(a.ws.xscale + threadIdx.x);
  for (int t = 0; t < a.T; ++t)
    topk_block(a.ws.logits + (size_t)t * a.E, a.bias, a.E, a.k, ku, sg, cand, a.ws.idx + (size_t)t * a.k,
               a.ws.w + (size_t)t * a.k, sidx + (size_t)t * a.k, sw + (size_t)t * a.k);
  if (P <= 32 && a.T <= kUnitTokens) {
    // few picks: one warp; the per-expert counts only when the tensor-core FFN follows
    if (threadIdx.x < 32)
      bucket_warp(sidx, sw, P, a.k, a.ws.perm, a.ws.act, a.ws.nact, a.ws.units, a.ws.nunits, sxs, bsm);
    if (a.need_counts) {
      __syncthreads();
      counts_from_sorted(bsm, P, a.E, a.ws.counts, a.ws.offsets);
    }
  } else if (P <= (int)blockDim.x && a.T <= kUnitTokens)
    bucket_small(sidx, sw, P, a.k, a.E, a.ws.counts, a.ws.offsets, a.ws.perm, a.ws.act, a.ws.nact, a.ws.units,
                 a.ws.nunits, sxs, bsm);
  else
    bucket_block(sidx, P, a.k, a.E, a.ws.counts, a.ws.offsets, a.ws.perm, a.ws.act, a.ws.nact, a.ws.units,
                 a.ws.nunits, sw, a.ws.xscale, bsm, true, true);
  if (threadIdx.x == 0) a.ws.sync[0] = 0u;
}

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float* logits, const float* bias, int T, int E, int k,
                                                            int32_t* idx, float* w) {
  extern __shared__ __align__(16) uint8_t tsm[];
  pdl_entry();
  uint32_t* ku = reinterpret_cast<uint32_t*>(tsm);
  float* sg = reinterpret_cast<float*>(ku + E);
  uint2* cand = reinterpret_cast<uint2*>(sg + E);  // word offset 2E: 8-byte aligned
  for (int t = blockIdx.x; t < T; t += gridDim.x)
    topk_block(logits + (size_t)t * E, bias, E, k, ku, sg, cand, idx + (size_t)t * k, w + (size_t)t * k);
}

constexpr int kWhistMaxE = 1536;  // 34 * E ints of shared memory (<= 204 KB)

__global__ void __launch_bounds__(1024) bucket_kernel(const int32_t* idx, int P, int k, int E, int32_t* counts,
                                                      int32_t* offsets, int32_t* perm, int32_t* act, int32_t* nact,
                                                      UnitDesc* units, int32_t* nunits, const float* w,
                                                      const float* xscale, int fill_units) {
  extern __shared__ int ism[];
  pdl_entry();
  int* whist = nullptr;
  if (E <= kWhistMaxE) {
    whist = ism + 2 * E;
    for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) whist[i] = 0;
  }
  bucket_block(idx, P, k, E, counts, offsets, perm, act, nact, units, nunits, w, xscale, ism, false, false, whist,
               fill_units != 0);
}

// ------------------------------------------------------------- multi-CTA bucketing ---
// For many picks (the tensor-core path and the bucketing entry point, which need counts,
// offsets and perm but no unit pick lists): chunk c = picks [c*kBkChunk, (c+1)*kBkChunk).
//   bucket_hist_kernel     chist[c][e] = picks of expert e in chunk c
//   bucket_scan_kernel     counts, offsets (exclusive scan over e), active list, unit count;
//                          chist[c][e] becomes offsets[e] + picks of e in chunks before c
//   bucket_scatter_kernel  chunk c's picks in pick order: perm[chist[c][e] + rank] = p, the rank
//                          counting earlier picks of e in the chunk (per-warp histograms)
// so perm lists every expert's picks in increasing pick id, as the single-block kernel does.
constexpr int kBkChunk = 2048;
constexpr int kBkThreads = 1024;
constexpr int kBkMultiMin = 4096;

__global__ void __launch_bounds__(kBkThreads) bucket_hist_kernel(const int32_t* idx, int P, int E, int32_t* chist) {
  extern __shared__ int hcnt[];
  pdl_entry();
  const int lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hcnt[e] = 0;
  __syncthreads();
  const int p0 = blockIdx.x * kBkChunk;
  for (int p = p0 + (int)threadIdx.x; p < p0 + kBkChunk; p += blockDim.x) {  // (uniform trip count)
    int e = p < P ? __ldcg(idx + p) : -1;
    if (e < 0 || e >= E) e = -1;
    const unsigned same = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && (same & ((1u << lane) - 1u)) == 0u) atomicAdd(&hcnt[e], __popc(same));
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chist[(size_t)blockIdx.x * E + e] = hcnt[e];
}

__global__ void __launch_bounds__(1024) bucket_scan_kernel(int32_t* chist, int C, int E, int32_t* counts,
                                                           int32_t* offsets, int32_t* act, int32_t* nact,
                                                           int32_t* nunits) {
  __shared__ int wsum[3][32];
  pdl_entry();
  const int tid = threadIdx.x, bd = blockDim.x, warp = tid >> 5, lane = tid & 31, nwarps = bd >> 5;
  // each thread owns a contiguous range of experts, so every output stays in expert-id order
  const int per = (E + bd - 1) / bd;
  const int ea = min(E, tid * per), eb = min(E, ea + per);
  int cs = 0, as = 0, us = 0;
  for (int e = ea; e < eb; ++e) {
    int v = 0;
    for (int c = 0; c < C; ++c) v += __ldcg(chist + (size_t)c * E + e);
    cs += v;
    as += v > 0;
    us += (v + kUnitTokens - 1) / kUnitTokens;
  }
  int ci = cs, ai = as, ui = us;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int c2 = __shfl_up_sync(0xffffffffu, ci, off), a2 = __shfl_up_sync(0xffffffffu, ai, off),
              u2 = __shfl_up_sync(0xffffffffu, ui, off);
    if (lane >= off) {
      ci += c2;
      ai += a2;
      ui += u2;
    }
  }
  if (lane == 31) {
    wsum[0][warp] = ci;
    wsum[1][warp] = ai;
    wsum[2][warp] = ui;
  }
  __syncthreads();
  if (warp == 0) {
    const int c0 = lane < nwarps ? wsum[0][lane] : 0, a0 = lane < nwarps ? wsum[1][lane] : 0,
              u0 = lane < nwarps ? wsum[2][lane] : 0;
    int cc = c0, aa = a0, uu = u0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int c2 = __shfl_up_sync(0xffffffffu, cc, off), a2 = __shfl_up_sync(0xffffffffu, aa, off),
                u2 = __shfl_up_sync(0xffffffffu, uu, off);
      if (lane >= off) {
        cc += c2;
        aa += a2;
        uu += u2;
      }
    }
    __syncwarp();
    if (lane < nwarps) {
      wsum[0][lane] = cc - c0;
      wsum[1][lane] = aa - a0;
      wsum[2][lane] = uu - u0;
    }
    if (lane == 31) {
      offsets[E] = cc;
      *nact = aa;
      *nunits = uu;
    }
  }
  __syncthreads();
  int run = wsum[0][warp] + ci - cs, arun = wsum[1][warp] + ai - as;
  for (int e = ea; e < eb; ++e) {
    const int start = run;
    for (int c = 0; c < C; ++c) {  // chunk bases in place
      const size_t at = (size_t)c * E + e;
      const int v = __ldcg(chist + at);
      chist[at] = run;
      run += v;
    }
    offsets[e] = start;
    counts[e] = run - start;
    if (run > start) act[arun++] = e;
  }
}

__global__ void __launch_bounds__(kBkThreads) bucket_scatter_kernel(const int32_t* idx, int P, int E,
                                                                    const int32_t* chist, int32_t* perm) {
  extern __shared__ int ssm[];
  int* cur = ssm;            // [E] next free position of each expert for this chunk
  int* whist = ssm + E;      // [32][E] picks of each expert in each warp of the current round
  pdl_entry();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int e = tid; e < E; e += blockDim.x) cur[e] = __ldcg(chist + (size_t)blockIdx.x * E + e);
  for (int i = tid; i < 32 * E; i += blockDim.x) whist[i] = 0;
  __syncthreads();
  const int p0 = blockIdx.x * kBkChunk;
  for (int r0 = p0; r0 < p0 + kBkChunk; r0 += blockDim.x) {  // (uniform trip count)
    const int p = r0 + tid;
    int e = p < P ? __ldcg(idx + p) : -1;
    const bool valid = e >= 0 && e < E;
    if (!valid) e = -1;
    const unsigned same = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(same & ((1u << lane) - 1u));
    if (valid && rank == 0) whist[warp * E + e] = __popc(same);
    __syncthreads();
    if (valid) {
      int base = cur[e];
      for (int w2 = 0; w2 < warp; ++w2) base += whist[w2 * E + e];
      perm[base + rank] = p;
    }
    __syncthreads();
    if (valid && rank == 0) {
      atomicAdd(&cur[e], __popc(same));
      whist[warp * E + e] = 0;
    }
    __syncthreads();
  }
}

}  // namespace

// x -> fp16 B fragments and the per-token power of two, one CTA per token at a time: the
// register-decode FFN's input when the logits come from the tensor-core router
__global__ void __launch_bounds__(kRouterWarps * 32) convert_kernel(RouterArgs a) {
  extern __shared__ __align__(16) uint8_t csm[];
  __shared__ float red[kRouterWarps];
  pdl_entry();
  uint16_t* xr = reinterpret_cast<uint16_t*>(csm);
  for (int t = blockIdx.x; t < a.T; t += gridDim.x) {
    __syncthreads();
    stage_tokens(a, t, 1, xr);
    __syncthreads();
    convert_token(a, t, xr, red);
  }
}

cudaError_t launch_convert(const RouterArgs& a, int num_sms, cudaStream_t s) {
  const int grid = std::min(a.T, 2 * num_sms);
  return launch_pdl(convert_kernel, dim3(grid), dim3(kRouterWarps * 32), (size_t)a.d * sizeof(uint16_t), s, a);
}

cudaError_t launch_router(const RouterArgs& a, cudaStream_t s) {
  // dynamic shared memory: the staged token tile, reused by the last block for top-k keys
  // (kRouterWarps * E floats) and bucketing (2 * E ints)
  size_t smem = (size_t)std::min(a.T, kTokTile) * a.d * sizeof(uint16_t);
  if (a.fuse_select) smem = std::max(smem, fused_select_smem(a.E, a.T * a.k));
  static std::atomic<unsigned long long> attr{0};
  const cudaError_t e = set_smem_limit_once(router_kernel, 200 * 1024, attr);
  if (e != cudaSuccess) return e;
  const int grid = (a.E + kRowsPerCta - 1) / kRowsPerCta;
  return launch_pdl(router_kernel, dim3(grid), dim3(kRouterWarps * 32), smem, s, a);
}

cudaError_t launch_topk(const float* logits, const float* bias, int T, int E, int k, int32_t* idx, float* w,
                        cudaStream_t s) {
  static std::atomic<unsigned long long> attr{0};
  const cudaError_t e = set_smem_limit_once(topk_kernel, 200 * 1024, attr);
  if (e != cudaSuccess) return e;
  const size_t smem = (size_t)(2 * E + 2) * 4 + 256 * 8;
  return launch_pdl(topk_kernel, dim3(std::min(T, 148 * 8)), dim3(kTopkThreads), smem, s, logits, bias, T, E, k, idx, w);
}

cudaError_t launch_bucket(const int32_t* idx, int T, int k, int E, int32_t* counts, int32_t* offsets,
                          int32_t* perm, int32_t* act, int32_t* nact, UnitDesc* units, int32_t* nunits,
                          const float* w, const float* xscale, int32_t* chist, cudaStream_t s, bool fill_units) {
  static std::atomic<unsigned long long> attr_b{0}, attr_s{0};
  cudaError_t e = set_smem_limit_once(bucket_kernel, 210 * 1024, attr_b);
  if (e == cudaSuccess) e = set_smem_limit_once(bucket_scatter_kernel, 210 * 1024, attr_s);
  if (e != cudaSuccess) return e;
  const int P = T * k;
  if (!fill_units && chist && P >= kBkMultiMin && E <= kWhistMaxE) {
    // many picks: histogram, scan and stable scatter spread over chunks of kBkChunk picks
    const int C = (P + kBkChunk - 1) / kBkChunk;
    e = launch_pdl(bucket_hist_kernel, dim3(C), dim3(kBkThreads), (size_t)E * sizeof(int), s, idx, P,
                               E, chist);
    if (e == cudaSuccess)
      e = launch_pdl(bucket_scan_kernel, dim3(1), dim3(1024), 0, s, chist, C, E, counts, offsets, act, nact, nunits);
    if (e == cudaSuccess)
      e = launch_pdl(bucket_scatter_kernel, dim3(C), dim3(kBkThreads), (size_t)33 * E * sizeof(int), s, idx, P, E,
                     (const int32_t*)chist, perm);
    return e;
  }
  const size_t smem = (size_t)(E <= kWhistMaxE ? 34 : 2) * E * sizeof(int);
  return launch_pdl(bucket_kernel, dim3(1), dim3(1024), smem, s, idx, T * k, k, E, counts, offsets, perm, act,
                    nact, units, nunits, w, xscale, fill_units ? 1 : 0);
}

}  // namespace k3
