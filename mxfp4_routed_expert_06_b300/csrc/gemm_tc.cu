// gemm_tc.cu -- large-T expert FFN as a grouped GEMM on the 5th-generation tensor cores.
//
// "kimi-k3-in-c deep dive", "four reductions", reduction 1: the experts stay MXFP4 (E2M1
// nibbles, one E8M0 scale per 32 values along the reduction axis) and are multiplied without
// a dense copy in memory.  With many tokens per expert the FFN is a dense contraction, so
// here each CTA decodes the weight tile it is about to use into shared memory (fp16, in the
// layout the tensor core reads) and multiplies it with tcgen05.mma, the fp32 accumulator
// living in tensor memory (TMEM).  Nothing is expanded in HBM.
//
// Numerics.  An E2M1 value is exact in fp16.  The block scale 2^(s-127) is split as
// 2^(s-s_ref) * 2^(s_ref-127): the first factor is multiplied into the fp16 weight (exact:
// a power of two, and the layer's scale bytes span at most 36 so that every decoded value is
// an fp16 number), the second is a per-layer constant applied to the fp32 accumulator.
// Activations enter as fp16 with one power-of-two factor per row (x per token, h per routed
// pick), so fp16 never overflows; h is kept in fp32 until its fp16 image is made (relative
// rounding 2^-11).  fp16 x fp16 products are exact and every sum is fp32.
//
// Kernels, in launch order (after routing and bucketing):
//   gemm_prep_x_kernel   per-token power of two of x (max |x| -> [2^14, 2^15) in fp16)
//   gemm_tiles_kernel    one M-tile descriptor per (expert, 128 consecutive picks of it)
//   gemm_gather_kernel   xg[row] = fp16 image of x[token of row], rows in bucketed order
//   gemm_kernel<GU>      [picks of e] x [gate|up rows of e]^T, SwiGLU in the epilogue,
//                        h -> fp32 [P][f] (bucketed row order) + max |h| per row
//   gemm_h16_kernel      h fp32 -> fp16 with a power of two per row
//   gemm_kernel<DN>      [picks of e] x [down rows of e]^T, times the combine weight,
//                        -> obuf[pick][d]; the combine kernel then sums the k slots in order.
//
// gemm_kernel is persistent (one CTA per SM).  A work item is (two consecutive 128-row M-tiles
// of one expert, N tile): every decoded weight stage feeds the MMAs of both M-tiles, which
// halves the decode work per flop.  Warp roles:
//   warps 0-3   epilogue: TMEM -> registers (warp w reads TMEM lanes 32w..32w+31 = tile rows)
//   warp  4     TMEM allocation; lane 0 issues the MMAs (M=128, N=256 or 128, K=16 each; the two
//               M-tiles accumulate in TMEM columns 0.. and 256..)
//   warp  5     lane 0 issues the 2-D TMA loads of the item's activation rows per stage
//               (rows are contiguous: xg for GU, h16 for DN, both in bucketed order)
//   warps 6-13  B decoders: MXFP4 bytes (registers, prefetched 4 stages ahead) ->
//               cvt e2m1x2 -> f16x2, times 2^(s-s_ref) -> shared memory
// A stage is 64 values of K: A 2 x 128x64 fp16 (2 x 16 KB) + B up to 256x64 fp16 (32 KB), all
// K-major with the 128-byte swizzle; 3 stages.  The epilogue drains both accumulators before
// the next item's MMAs start.  Every wait is bounded (globaltimer).
#include <cuda.h>
#include <cuda_bf16.h>

#include "k3moe_internal.cuh"

namespace k3 {
namespace {

// ------------------------------------------------------------------- PTX helpers ---
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait on the phase of parity `parity`.  false: gave up (error flag set) or another
// thread already reported an error.
__device__ __noinline__ bool wait_phase(uint64_t* bar, uint32_t parity, uint32_t* err, unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = now_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0u) {
      if (*reinterpret_cast<volatile uint32_t*>(err) != 0u) return false;
      if (now_ns() - t0 > limit_ns) {
        atomicOr(err, kErrTimeout);
        return false;
      }
    }
  }
}

// Bounded wait that ignores the error flag: for the final MMA drain, which always completes
// (the MMAs in flight read only shared memory that is already written).
__device__ __noinline__ bool wait_phase_drain(uint64_t* bar, uint32_t parity, uint32_t* err,
                                              unsigned long long limit_ns) {
  const unsigned long long t0 = now_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 255u && now_ns() - t0 > limit_ns) {
      atomicOr(err, kErrTimeout);
      return false;
    }
  }
}

// The barrier's current phase also waits for `bytes` of asynchronous (TMA) writes.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
// 2-D tiled TMA load of the box at (c0 = inner element, c1 = row); completes on `bar`.
// c0 * 2 bytes is a multiple of 16 (c0 is a multiple of 64), as every tiled TMA copy needs.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}
// generic-proxy writes to shared memory -> visible to the tensor core (async proxy)
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// tcgen05: TMEM allocation, MMA, commit, loads, fences
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// D[tmem] (+)= A[smem] * B[smem]^T, both K-major; accumulate = 0 overwrites D
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// the mbarrier completes one arrival when every MMA this thread issued before has finished
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
// 32 consecutive fp32 columns of the warp's 32 TMEM lanes (one row per thread)
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 bytes apart.
//   bits 0-13 start address >> 4; 16-29 leading byte offset >> 4 (unused for this layout: 1);
//   32-45 stride byte offset >> 4 (1024 B); 46-48 fixed 0b001; 49-51 base offset (0: tiles are
//   1024-byte aligned); 61-63 swizzle mode (2 = 128-byte).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B fp16 (bits 7-9, 10-12 = 0),
// both K-major (bits 15, 16 = 0), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// same with A and B bf16 (bits 7-9 and 10-12 = 1)
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) { return idesc_f16(M, N) | (1u << 7) | (1u << 10); }

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
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// fp16 bits of 2^e for -24 <= e <= 15 (subnormal below -14), both halves of a word
__device__ __forceinline__ uint32_t pow2_h2(int e) {
  const uint32_t h = e >= -14 ? (uint32_t)(e + 15) << 10 : 1u << (e + 24);
  return h | (h << 16);
}

// power-of-two exponent q with m * 2^-q in [2^14, 2^15): the fp16 image never overflows
__device__ __forceinline__ int fp16_scale_exp(float m) {
  if (!(m > 0.0f)) return 0;
  const int ex = (int)((__float_as_uint(m) >> 23) & 0xFFu) - 127;
  const int q = ex - 14;
  return q < -126 ? -126 : (q > 126 ? 126 : q);
}
__device__ __forceinline__ float exp2i(int q) { return __uint_as_float((uint32_t)(127 + q) << 23); }

// ----------------------------------------------------------------------- constants ---
constexpr int kStages = 3;
constexpr int kBM = 128;                 // rows (picks) per M-tile; a work item has two
constexpr int kBK = 64;                  // K values per stage
constexpr int kABytes = kBM * kBK * 2;   // 16 KB per M-tile
constexpr int kBBytes = 256 * kBK * 2;   // 32 KB (N up to 256)
constexpr int kStageBytes = 2 * kABytes + kBBytes;  // A of both M-tiles, then B
constexpr int kEpiWarps = 4;
constexpr int kMmaWarp = 4;
constexpr int kTmaWarp = 5;
constexpr int kDecWarp0 = 6;
constexpr int kDecWarps = 8;
constexpr int kGemmThreads = (kDecWarp0 + kDecWarps) * 32;  // 448
constexpr int kTmemCols = 512;           // accumulators of the two M-tiles, up to 256 fp32 columns each
constexpr int kPf = 4;                   // B decoders: stages of raw bytes held in registers
// shared memory: stages, then barriers; +1024 for alignment
constexpr size_t kGemmSmem = 1024 + (size_t)kStages * kStageBytes + 256;

struct GemmArgs {
  const uint8_t* const* expert_ptr;
  int d, f, k, T;
  int mode;                 // 0: gate/up + SwiGLU, 1: down, 2: router logits
  int E;                    // router: experts (B rows)
  float* logits;            // router output [T][E]
  int bn;                   // N of a work item: 256 (GU: 128 gate + 128 up rows; DN: 256 rows) or 128 (DN)
  int s_ref;
  float wscale;             // 2^(s_ref - 127)
  const int4* mtiles;       // {expert, first bucketed row, rows of M-tile 0, rows of M-tile 1}
  const int32_t* nmtiles;
  const int32_t* perm;      // bucketed row -> pick id
  const float* wgt;         // [P] combine weights by pick
  const float* ascale;      // GU: x power of two [T]; DN: h power of two [P] (bucketed rows)
  float* hbuf;              // GU output [P][f]
  uint32_t* hmax;           // GU output [P] (float bits of max |h|)
  float* obuf;              // DN output [P][d] by pick
  uint32_t* err;
  unsigned long long wait_ns;
  int act;                  // gate activation (K3MOE_ACT_*), mode 0
};

// Raw bytes one decoder lane needs for one stage: two tile halves (16 nibble bytes each) and
// their scale words (rows g and g+8 x 4 blocks).
struct Raw {
  uint4 n0, n1;
  uint2 s0, s1;
};

// Work item i = (pair of M-tiles i / NT, N tile i % NT).  The pair: two consecutive 128-row
// M-tiles of one expert (the second may be empty); for the router, 256 consecutive tokens.
struct Pair {
  int e, row0, rows0, rows1;
};
template <int MODE>
__device__ __forceinline__ Pair pair_of(const GemmArgs& a, int pt) {
  if (MODE == 2) {
    const int row0 = pt * 2 * kBM;
    return Pair{0, row0, min(kBM, a.T - row0), max(0, min(kBM, a.T - row0 - kBM))};
  }
  const int4 v = __ldg(a.mtiles + pt);
  return Pair{v.x, v.y, v.z, v.w};
}

// tmap_a: 2-D map of the activation rows (fp16 [P][K], or bf16 x [T][d] for the router; box
// 64 x 128, 128-byte swizzle).  tmap_b (router only): W_r split into bf16 hi and lo halves,
// [E][2d], box 64 x 128.
template <int MODE>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b, GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* accf = empty + kStages;  // [2] accumulators of buffer b ready
  uint64_t* acce = accf + 2;         // [2] accumulators of buffer b drained by the epilogue
  uint64_t* drain = acce + 2;        // final MMA completion
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], MODE == 2 ? 1 : 1 + kDecWarps);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], kEpiWarps);
    }
    mbar_init(drain, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_entry();  // set-up above touched only shared and tensor memory

  // router: K runs over [x | x] against [W_hi | W_lo], i.e. 2d values
  const int K = MODE == 0 ? a.d : (MODE == 1 ? a.f : 2 * a.d);
  const int KS = K / kBK;
  const int KSh = a.d / kBK;
  const int KT = K / kTileCols;
  const int NT = MODE == 0 ? a.f / (a.bn / 2) : (MODE == 1 ? a.d / a.bn : (a.E + 127) / 128);
  // N <= 128: two accumulator buffers (2 M-tiles x 128 columns each) so that the epilogue of one
  // item overlaps the next item's MMAs; N = 256: one buffer of 2 x 256 columns
  const int nbuf = a.bn <= 128 ? 2 : 1;
  const int n_items = (MODE == 2 ? (a.T + 2 * kBM - 1) / (2 * kBM) : *a.nmtiles) * NT;
  const int G = gridDim.x;
  const uint32_t sbase = smem_u32(smem);

  if (warp < kEpiWarps) {
    // ------------------------------------------------------------------ epilogue ---
    int it = 0;
    for (int i = blockIdx.x; i < n_items; i += G, ++it) {
      const int buf = it % nbuf, use = it / nbuf;
      if (!wait_phase(&accf[buf], (uint32_t)(use & 1), a.err, a.wait_ns)) break;
      tc_fence_after();
      const int nt = i % NT;
      const Pair pr = pair_of<MODE>(a, i / NT);
      const int r = warp * 32 + lane;
      for (int h = 0; h < 2; ++h) {
        const int rows = h ? pr.rows1 : pr.rows0;
        if (rows <= 0) continue;  // uniform across the warp
        const uint32_t tb = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(buf * 256 * (nbuf - 1) + h * a.bn);
        const bool valid = r < rows;
        const int pos = pr.row0 + h * kBM + (valid ? r : 0);
        if (MODE == 2) {
          const int c0 = nt * 128;
          float* dst = a.logits + (size_t)pos * a.E + c0;
          for (int c = 0; c < 4; ++c) {
            uint32_t v[32];
            tmem_ld32(tb + 32 * c, v);
            tmem_ld_wait();
            if (valid) {
              if ((a.E & 3) == 0 && c0 + 32 * c + 32 <= a.E) {
                float4* d4 = reinterpret_cast<float4*>(dst + 32 * c);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                  d4[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                      __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  if (c0 + 32 * c + j < a.E) dst[32 * c + j] = __uint_as_float(v[j]);
              }
            }
          }
          continue;
        }
        const int p = __ldg(a.perm + pos);
        if (MODE == 0) {
          const float sc = __ldg(a.ascale + p / a.k) * a.wscale;
          float mx = 0.f;
          const int half = a.bn / 2;  // gate columns [0, half), up columns [half, bn)
          float* dst = a.hbuf + (size_t)pos * a.f + nt * half;
          for (int c = 0; c < half / 32; ++c) {
            uint32_t gr[32], ur[32];
            tmem_ld32(tb + 32 * c, gr);
            tmem_ld32(tb + half + 32 * c, ur);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float g = __uint_as_float(gr[j]) * sc, u = __uint_as_float(ur[j]) * sc;
              const float hv = gate_act(g, a.act) * u;
              gr[j] = __float_as_uint(hv);
              mx = fmaxf(mx, fabsf(hv));
            }
            if (valid) {
              float4* d4 = reinterpret_cast<float4*>(dst + 32 * c);
#pragma unroll
              for (int q = 0; q < 8; ++q)
                d4[q] = make_float4(__uint_as_float(gr[4 * q]), __uint_as_float(gr[4 * q + 1]),
                                    __uint_as_float(gr[4 * q + 2]), __uint_as_float(gr[4 * q + 3]));
            }
          }
          if (valid) atomicMax(a.hmax + pos, __float_as_uint(mx));
        } else {
          const float sc = __ldg(a.ascale + pos) * a.wscale * __ldg(a.wgt + p);
          float* dst = a.obuf + (size_t)p * a.d + (size_t)nt * a.bn;
          for (int c = 0; c < a.bn / 32; ++c) {
            uint32_t orr[32];
            tmem_ld32(tb + 32 * c, orr);
            tmem_ld_wait();
            if (valid) {
              float4* d4 = reinterpret_cast<float4*>(dst + 32 * c);
#pragma unroll
              for (int q = 0; q < 8; ++q)
                d4[q] = make_float4(__uint_as_float(orr[4 * q]) * sc, __uint_as_float(orr[4 * q + 1]) * sc,
                                    __uint_as_float(orr[4 * q + 2]) * sc, __uint_as_float(orr[4 * q + 3]) * sc);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce[buf]);
    }
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------------- MMA issue ---
    if (lane == 0) {
      const uint32_t idesc = MODE == 2 ? idesc_bf16(kBM, 128) : idesc_f16(kBM, a.bn);
      uint32_t g = 0;
      int it = 0;
      bool ok = true;
      for (int i = blockIdx.x; i < n_items && ok; i += G, ++it) {
        const bool two = pair_of<MODE>(a, i / NT).rows1 > 0;
        const int buf = it % nbuf, use = it / nbuf;
        if (!wait_phase(&acce[buf], (uint32_t)((use & 1) ^ 1), a.err, a.wait_ns)) break;
        const uint32_t d0 = tmem + (uint32_t)(buf * 256 * (nbuf - 1)), d1 = d0 + (uint32_t)a.bn;
        tc_fence_after();
        for (int ks = 0; ks < KS; ++ks, ++g) {
          const int slot = (int)(g % kStages);
          if (!wait_phase(&full[slot], (g / kStages) & 1u, a.err, a.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t as = sbase + (uint32_t)(slot * kStageBytes);
          const uint64_t a0 = smem_desc(as), a1 = smem_desc(as + kABytes), bd = smem_desc(as + 2 * kABytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {  // +32 bytes along K per k16 step
            const uint32_t accum = (ks | kk) != 0 ? 1u : 0u;
            mma_f16(d0, a0 + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), idesc, accum);
            if (two) mma_f16(d1, a1 + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), idesc, accum);
          }
          mma_commit(&empty[slot]);
        }
        if (ok) mma_commit(&accf[buf]);
      }
      // everything issued has completed before TMEM is released
      mma_commit(drain);
      wait_phase_drain(drain, 0, a.err, a.wait_ns);
    }
    __syncwarp();
  } else if (warp == kTmaWarp) {
    // ------------------------------------------------------------- A (TMA) issue ---
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
      if (MODE == 2) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_b)) : "memory");
      uint32_t g = 0;
      bool ok = true;
      for (int i = blockIdx.x; i < n_items && ok; i += G) {
        const Pair pr = pair_of<MODE>(a, i / NT);
        const bool two = pr.rows1 > 0;
        for (int ks = 0; ks < KS; ++ks, ++g) {
          const int slot = (int)(g % kStages);
          if (!wait_phase(&empty[slot], ((g / kStages) & 1u) ^ 1u, a.err, a.wait_ns)) {
            ok = false;
            break;
          }
          const uint32_t st = sbase + (uint32_t)(slot * kStageBytes);
          const int kc = MODE == 2 ? (ks % KSh) * kBK : ks * kBK;
          const uint32_t bytes = (uint32_t)kABytes * (two ? 2u : 1u) + (MODE == 2 ? 128u * kBK * 2u : 0u);
          mbar_arrive_expect_tx(&full[slot], bytes);
          tma_load_2d(st, &tmap_a, kc, pr.row0, &full[slot]);
          if (two) tma_load_2d(st + kABytes, &tmap_a, kc, pr.row0 + kBM, &full[slot]);
          if (MODE == 2) tma_load_2d(st + 2 * kABytes, &tmap_b, ks * kBK, (i % NT) * 128, &full[slot]);
        }
      }
      // no load may be in flight when the CTA exits: the last use of each slot has completed
      // (normally the MMAs already waited for it)
      for (uint32_t q = g > (uint32_t)kStages ? g - kStages : 0; q < g; ++q)
        wait_phase_drain(&full[q % kStages], (q / kStages) & 1u, a.err, a.wait_ns);
    }
    __syncwarp();
  } else if (MODE != 2) {
    // ---------------------------------------------------------------- B decoders ---
    const int dw = warp - kDecWarp0;
    const int gq = lane >> 2, tq = lane & 3;
    const int my_items = (int)blockIdx.x < n_items ? (n_items - (int)blockIdx.x + G - 1) / G : 0;
    const int total = my_items * KS;
    const size_t gu_bytes = gateup_region_bytes(a.d, a.f);
    const int groups = a.bn / 16;  // 16-row groups of B per stage
    // Fetch cursor: the stage whose bytes are loaded next (stages are fetched in order).  The
    // item's tile addresses are recomputed only when the cursor enters a new item.
    int c_li = 0, c_ks = 0;
    const uint8_t* c_t0 = nullptr;  // tile of half 0 at k-tile 0 of the cursor's item
    const uint8_t* c_t1 = nullptr;  // half 1 (nullptr when unused)
    auto enter_item = [&]() {
      const int i = (int)blockIdx.x + c_li * G;
      if (i >= n_items) return;
      const int mt = i / NT, nt = i % NT;
      const uint8_t* base = a.expert_ptr[__ldg(&a.mtiles[mt].x)];
      if (MODE == 0) {
        if (groups == 16) {  // N = 256: gate rows 16dw.. and up rows 128+16dw.. of row group nt*8+dw
          c_t0 = base + (size_t)(nt * 8 + dw) * KT * 2 * kTileBytes;
          c_t1 = c_t0 + kTileBytes;
        } else {  // N = 128: warps 0-3 take gate row groups nt*4+dw, warps 4-7 the matching up tiles
          c_t0 = base + (size_t)(nt * 4 + (dw & 3)) * KT * 2 * kTileBytes + (dw >= 4 ? kTileBytes : 0);
          c_t1 = nullptr;
        }
      } else {
        c_t0 = base + gu_bytes + (size_t)(nt * groups + dw) * KT * kTileBytes;
        c_t1 = dw + 8 < groups ? c_t0 + (size_t)8 * KT * kTileBytes : nullptr;
      }
    };
    const size_t kt_stride = MODE == 0 ? 2 * (size_t)kTileBytes : (size_t)kTileBytes;
    enter_item();
    auto fetch = [&](int s, Raw& r) {
      if (s >= total) return;
      const int u = c_ks & 1;
      const size_t off = (size_t)(c_ks >> 1) * kt_stride;
      const uint8_t* t0 = c_t0 + off;
      r.n0 = __ldg(reinterpret_cast<const uint4*>(t0 + u * 512 + lane * 16));
      r.s0 = __ldg(reinterpret_cast<const uint2*>(t0 + kTileNibBytes + gq * 8));
      if (c_t1) {
        const uint8_t* t1 = c_t1 + off;
        r.n1 = __ldg(reinterpret_cast<const uint4*>(t1 + u * 512 + lane * 16));
        r.s1 = __ldg(reinterpret_cast<const uint2*>(t1 + kTileNibBytes + gq * 8));
      }
      if (++c_ks == KS) {
        c_ks = 0;
        ++c_li;
        enter_item();
      }
    };
    // decode one tile half into B rows n0 .. n0+15 of the stage at byte address bs
    auto decode = [&](const uint4& nib, const uint2& sc, int u, int n0, uint32_t bs) {
      // scale bytes of rows gq (sc.x) and gq+8 (sc.y), blocks 2u and 2u+1
      uint32_t f[2][2];
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
          const uint32_t w4 = h ? sc.y : sc.x;
          const int s8 = (int)((w4 >> (8 * (2 * u + bb))) & 0xFFu);
          f[h][bb] = pow2_h2(s8 - a.s_ref);
        }
      const uint32_t rowA = bs + (uint32_t)((n0 >> 3) * 1024 + gq * 128);  // row n0+gq
      const uint32_t rowB = rowA + 1024;                                     // row n0+gq+8
      const uint32_t words[4] = {nib.x, nib.y, nib.z, nib.w};
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        uint32_t v[4];
        dec4(words[s], v);
        const int bb = s >> 1;
        const uint32_t c0 = (uint32_t)((((2 * s) ^ gq) << 4) + 4 * tq);
        const uint32_t c1 = (uint32_t)((((2 * s + 1) ^ gq) << 4) + 4 * tq);
        sts32(rowA + c0, hmul2(v[0], f[0][bb]));
        sts32(rowB + c0, hmul2(v[1], f[1][bb]));
        sts32(rowA + c1, hmul2(v[2], f[0][bb]));
        sts32(rowB + c1, hmul2(v[3], f[1][bb]));
      }
    };
    Raw raw[kPf];
#pragma unroll
    for (int j = 0; j < kPf; ++j) fetch(j, raw[j]);
    bool ok = true;
    for (int s0 = 0; s0 < total && ok; s0 += kPf) {
#pragma unroll
      for (int j = 0; j < kPf; ++j) {
        const int s = s0 + j;
        if (s < total && ok) {
          const uint32_t g = (uint32_t)s;
          const int slot = (int)(g % kStages);
          if (!wait_phase(&empty[slot], ((g / kStages) & 1u) ^ 1u, a.err, a.wait_ns)) {
            ok = false;
          } else {
            const int u = (s % KS) & 1;
            const uint32_t bs = sbase + (uint32_t)(slot * kStageBytes + 2 * kABytes);
            if (MODE == 0 && groups == 16) {
              decode(raw[j].n0, raw[j].s0, u, 16 * dw, bs);        // gate rows
              decode(raw[j].n1, raw[j].s1, u, 128 + 16 * dw, bs);  // up rows
            } else if (MODE == 0) {
              decode(raw[j].n0, raw[j].s0, u, (dw >= 4 ? 64 : 0) + 16 * (dw & 3), bs);
            } else {
              decode(raw[j].n0, raw[j].s0, u, 16 * dw, bs);
              if (dw + 8 < groups) decode(raw[j].n1, raw[j].s1, u, 16 * (dw + 8), bs);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&full[slot]);
            fetch(s + kPf, raw[j]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------- small kernels ---

// per-token power of two: xs[t] = 2^q with max|x_t| * 2^-q in [2^14, 2^15)
__global__ void __launch_bounds__(256) gemm_prep_x_kernel(const uint16_t* __restrict__ x, int d, float* xs) {
  pdl_entry();
  __shared__ float part[8];
  const size_t base = (size_t)blockIdx.x * d;
  float mx = 0.f;
  for (int j = threadIdx.x; j < d; j += 256) mx = fmaxf(mx, fabsf(__uint_as_float((uint32_t)x[base + j] << 16)));
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < 8; ++w) mx = fmaxf(mx, part[w]);
    mx = fmaxf(mx, part[0]);
    xs[blockIdx.x] = exp2i(fp16_scale_exp(mx));
  }
}

// xg[row] = fp16(x[t] / xs[t]), t = token of the pick at bucketed row `row` (one CTA per row)
__global__ void __launch_bounds__(128) gemm_gather_kernel(const uint16_t* __restrict__ x, const float* __restrict__ xs,
                                                          const int32_t* __restrict__ perm, int d, int k,
                                                          __half* __restrict__ xg) {
  pdl_entry();
  const int t = __ldg(perm + blockIdx.x) / k;
  const float inv = 1.0f / __ldg(xs + t);  // a power of two: exact
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d);
  uint4* dst = reinterpret_cast<uint4*>(xg + (size_t)blockIdx.x * d);
  for (int v = threadIdx.x; v < d / 8; v += 128) {
    const uint4 b = __ldg(src + v);
    const uint32_t w[4] = {b.x, b.y, b.z, b.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float lo = __uint_as_float(w[q] << 16) * inv, hi = __uint_as_float(w[q] & 0xFFFF0000u) * inv;
      o[q] = (uint32_t)__half_as_ushort(__float2half_rn(lo)) | ((uint32_t)__half_as_ushort(__float2half_rn(hi)) << 16);
    }
    dst[v] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// M-tile pairs: for each expert e (ascending) ceil(count/256) pairs of 128-row tiles of
// consecutive bucketed rows (the second tile of the last pair may be short or empty)
__global__ void __launch_bounds__(1024) gemm_tiles_kernel(const int32_t* __restrict__ counts,
                                                          const int32_t* __restrict__ offsets, int E, int4* mtiles,
                                                          int32_t* nmtiles) {
  pdl_entry();
  __shared__ int wsum[32];
  const int per = (E + 1023) / 1024;
  const int e0 = threadIdx.x * per;
  int local = 0;
  for (int e = e0; e < min(E, e0 + per); ++e) local += (counts[e] + 2 * kBM - 1) / (2 * kBM);
  // block exclusive scan
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = local;
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int v = wsum[lane];
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    wsum[lane] = v;
  }
  __syncthreads();
  int start = incl - local + (warp > 0 ? wsum[warp - 1] : 0);
  for (int e = e0; e < min(E, e0 + per); ++e) {
    const int c = counts[e], o = offsets[e];
    for (int r0 = 0; r0 < c; r0 += 2 * kBM)
      mtiles[start++] = make_int4(e, o + r0, min(kBM, c - r0), max(0, min(kBM, c - r0 - kBM)));
  }
  if (threadIdx.x == 1023) *nmtiles = start;
}

// h fp32 -> h16 fp16 with one power of two per row (h = h16 * hs[row])
__global__ void __launch_bounds__(256) gemm_h16_kernel(const float* __restrict__ hbuf, uint32_t* hmax, int f,
                                                       __half* h16,
                                                       float* hs) {
  pdl_entry();
  const size_t base = (size_t)blockIdx.x * f;
  const int q = fp16_scale_exp(__uint_as_float(hmax[blockIdx.x]));
  const float inv = exp2i(-q);
  for (int j = threadIdx.x; j < f; j += 256) h16[base + j] = __float2half_rn(hbuf[base + j] * inv);
  __syncthreads();
  if (threadIdx.x == 0) {
    hs[blockIdx.x] = exp2i(q);
    hmax[blockIdx.x] = 0u;  // zero between calls (the register-decode path also accumulates into it)
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver (looked up once; the library does not link libcuda)
EncodeTiledFn encode_tiled() {
  static const EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return (EncodeTiledFn) nullptr;
    }
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// 16-bit [rows][K] row-major, boxes of 64 x 128 with the 128-byte swizzle the MMA descriptors use
cudaError_t activation_map(CUtensorMap* m, const void* base, int K, int rows,
                           CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_FLOAT16) {
  const EncodeTiledFn fn = encode_tiled();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kBM};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, type, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int MODE>
cudaError_t launch_gemm_mode(const CUtensorMap& map, const CUtensorMap& map_b, const GemmArgs& g, int grid,
                             cudaStream_t s) {
  static std::atomic<unsigned long long> attr{0};
  const cudaError_t e = set_smem_limit_once(gemm_kernel<MODE>, (int)kGemmSmem, attr);
  if (e != cudaSuccess) return e;
  return launch_pdl(gemm_kernel<MODE>, dim3(grid), dim3(kGemmThreads), kGemmSmem, s, map, map_b, g);
}

}  // namespace

bool gemm_scales_ok(int s_min, int s_max) { return s_max >= s_min && s_max - s_min <= 36; }

cudaError_t launch_gemm_prep(const GemmFfn& q, const uint16_t* x, const int32_t* counts, const int32_t* offsets,
                             int E, cudaStream_t s) {
  cudaError_t e = launch_pdl(gemm_prep_x_kernel, dim3(q.T), dim3(256), 0, s, x, q.d, q.xs);
  if (e != cudaSuccess) return e;
  e = launch_pdl(gemm_tiles_kernel, dim3(1), dim3(1024), 0, s, counts, offsets, E, const_cast<int4*>(q.mtiles),
                 const_cast<int32_t*>(q.nmtiles));
  if (e != cudaSuccess) return e;
  return launch_pdl(gemm_gather_kernel, dim3(q.T * q.k), dim3(128), 0, s, x, (const float*)q.xs, (const int32_t*)q.perm,
                    q.d, q.k, q.xg);
}

namespace {
GemmArgs common_args(const GemmFfn& q, int mode) {
  GemmArgs g{};
  g.expert_ptr = q.expert_ptr;
  g.d = q.d;
  g.f = q.f;
  g.k = q.k;
  g.T = q.T;
  g.mode = mode;
  g.s_ref = q.s_ref;
  g.wscale = q.wscale;
  g.mtiles = q.mtiles;
  g.nmtiles = q.nmtiles;
  g.perm = q.perm;
  g.wgt = q.w;
  g.err = q.err;
  g.wait_ns = q.wait_ns;
  g.act = q.act;
  return g;
}
}  // namespace

cudaError_t launch_gemm_gu(const GemmFfn& q, cudaStream_t s) {
  GemmArgs g = common_args(q, 0);
  // N = 256 (128 gate + 128 up rows per item, one accumulator buffer of 2 x 256 columns):
  // N = 128 with two buffers overlaps the epilogue but halves the MMA work per decoded
  // stage, which measured slower (gate/up 3.75 vs 2.78 ms on the K3 prefill)
  g.bn = 256;
  g.ascale = q.xs;
  g.hbuf = q.hbuf;
  g.hmax = q.hmax;
  CUtensorMap map;
  cudaError_t e = activation_map(&map, q.xg, q.d, q.T * q.k);
  if (e != cudaSuccess) return e;
  return launch_gemm_mode<0>(map, map, g, q.num_sms, s);
}

cudaError_t launch_gemm_h16(const GemmFfn& q, int P, cudaStream_t s) {
  return launch_pdl(gemm_h16_kernel, dim3(P), dim3(256), 0, s, (const float*)q.hbuf, q.hmax, q.f, q.h16, q.hs);
}

cudaError_t launch_gemm_dn(const GemmFfn& q, cudaStream_t s) {
  GemmArgs g = common_args(q, 1);
  g.bn = q.d % 256 == 0 ? 256 : 128;  // N = 256 measured faster than double-buffered N = 128
  g.ascale = q.hs;
  g.obuf = q.obuf;
  CUtensorMap map;
  cudaError_t e = activation_map(&map, q.h16, q.f, q.T * q.k);
  if (e != cudaSuccess) return e;
  return launch_gemm_mode<1>(map, map, g, q.num_sms, s);
}

cudaError_t launch_router_tc(const uint16_t* x, int T, int d, int E, const uint16_t* wsplit, float* logits,
                             uint32_t* err, unsigned long long wait_ns, int num_sms, cudaStream_t s) {
  GemmArgs g{};
  g.d = d;
  g.T = T;
  g.E = E;
  g.mode = 2;
  g.bn = 128;
  g.logits = logits;
  g.err = err;
  g.wait_ns = wait_ns;
  CUtensorMap ma, mb;
  cudaError_t e = activation_map(&ma, x, d, T, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
  if (e == cudaSuccess) e = activation_map(&mb, wsplit, 2 * d, E, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
  if (e != cudaSuccess) return e;
  const int items = (T + 2 * kBM - 1) / (2 * kBM) * ((E + 127) / 128);
  return launch_gemm_mode<2>(ma, mb, g, items < num_sms ? items : num_sms, s);
}

// W_r fp32 [E][d] -> [E][2d] bf16: W_hi = bf16(W) then W_lo = bf16(W - W_hi)
__global__ void split_router_kernel(const float* __restrict__ W, int E, int d, uint16_t* __restrict__ out) {
  const size_t n = (size_t)E * d;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const size_t e = i / d, j = i % d;
    const float w = W[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const __nv_bfloat16 lo = __float2bfloat16_rn(w - __bfloat162float(hi));
    out[e * 2 * d + j] = __bfloat16_as_ushort(hi);
    out[e * 2 * d + d + j] = __bfloat16_as_ushort(lo);
  }
}

cudaError_t launch_split_router(const float* W, int E, int d, uint16_t* out, cudaStream_t s) {
  split_router_kernel<<<1184, 256, 0, s>>>(W, E, d, out);
  return cudaGetLastError();
}

}  // namespace k3
