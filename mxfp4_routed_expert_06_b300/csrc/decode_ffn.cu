// decode_ffn.cu -- small-T expert FFN straight from the MXFP4 bytes (register decode).
//
// "kimi-k3-in-c deep dive", "four reductions", reduction 1: the experts stay MXFP4 and are
// multiplied on the nibbles, never expanded to a dense copy (value = E2M1[nibble] *
// 2^(scale-127), 32 values per scale).  Here every routed expert's bytes stream from HBM once
// per call into shared memory (per-warp cp.async rings, L2 evict-first), and consumer warps
// turn each byte into an f16x2 tensor-core
// fragment with the hardware e2m1x2 -> f16x2 conversion and multiply with mma.m16n8k16,
// the routed tokens of one work unit (<= 8) being the n = 8 columns.  The E8M0 scale of each
// 32-column block is applied once per block in fp32: the block's two k16 steps accumulate
// into a zeroed fp32 fragment that is added, times the scale, to the running sum.  fp16 x
// fp16 products are exact and every sum is fp32.
//
// Both FFN kernels are persistent (two CTAs per SM); a CTA walks tasks
// i = blockIdx.x + j*gridDim.x.  Each consumer warp streams its own stages from HBM with
// cp.async (16 bytes per lane, L2 evict-first) several stages ahead into a private shared-memory
// ring; on this GPU that keeps ~7 TB/s in flight, where a single-thread bulk-copy producer is
// limited by a per-copy cost.
//   gateup_kernel  task = (unit, 16 rows of f); stage = one 128-column k-tile of the gate and
//                  up tiles (2176 B) + the unit's x fragments for it; consumer warp w takes
//                  k-tiles kt % 8 == w; one of 2 epilogue warps adds the 8 partial sums in
//                  warp order, applies SwiGLU h = silu(g) * u (or SiTU-GLU, gate_act), writes
//                  h (fp32) and records max |h| per pick.
//   hconv_kernel   h -> fp16 B fragments with one power-of-two scale per pick (fp16 never
//                  overflows; the scale factors out of the down projection's sum).
//   down_kernel    task = (unit, 32 rows of d) over the whole f range, streamed in chunks of
//                  k-tiles; consumer warp = task % 8; writes w * hs * o to obuf[pick].
//   combine_kernel y[t] = sum over the k slots, in slot order, of obuf[t*k + slot].
// Every device-side wait is bounded (globaltimer); on expiry the kernel sets an error flag
// that the host reads at its next synchronisation, drains its copies in flight and returns.
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

// Bounded wait on one phase of an mbarrier.  false: the wait gave up (error flag set) or
// another thread of the grid already reported an error.
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

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ uint2 lds64(const uint8_t* p) { return *reinterpret_cast<const uint2*>(p); }

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

// Scale byte b (0..3) of a word of four E8M0 bytes, as fp32.  ZS = false when the layer has no
// zero scale byte (checked at pack time): then 2^(s-127) is just s placed in the exponent field.
template <bool ZS>
__device__ __forceinline__ float scale_of(uint32_t w4, int b) {
  const uint32_t s = __byte_perm(w4, 0u, 0x4440u + (uint32_t)b);
  return ZS ? e8m0f(s) : __uint_as_float(s << 23);
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int s) {
  return s == 0 ? v.x : (s == 1 ? v.y : (s == 2 ? v.z : v.w));
}

// power-of-two exponent q with m * 2^-q in [2^14, 2^15): the fp16 image never overflows
__device__ __forceinline__ int fp16_scale_exp(float m) {
  if (!(m > 0.0f)) return 0;
  const int ex = (int)((__float_as_uint(m) >> 23) & 0xFFu) - 127;
  const int q = ex - 14;
  return q < -126 ? -126 : (q > 126 ? 126 : q);
}
__device__ __forceinline__ float exp2i(int q) { return __uint_as_float((uint32_t)(127 + q) << 23); }

constexpr int kConsumers = 8;
constexpr int kStageAlign = 128;
constexpr int kMaxDepth = 6;  // outstanding cp.async groups per thread

// Asynchronous 16-byte global -> shared copy (L2 only) with an L2 eviction policy: expert bytes
// are read once per call and go evict-first, so that the router weights and the activations
// stay in L2 across calls.
#ifdef K3MOE_DEVICE_CHECKS
// Self-checking build: a misaligned or out-of-ring copy records kErrBadAccess and is skipped.
// Bounds are per CTA (shared-window offsets), set by thread 0 before the first copy.
__shared__ uint32_t g_chk_lo, g_chk_hi;
__shared__ uint32_t* g_chk_err;
#endif
__device__ __forceinline__ void cp16(void* dst, const void* src, uint64_t pol) {
#ifdef K3MOE_DEVICE_CHECKS
  const uint32_t d = smem_u32(dst);
  if ((d & 15u) != 0u || ((uintptr_t)src & 15u) != 0u || d < g_chk_lo || d + 16u > g_chk_hi) {
    atomicOr(g_chk_err, kErrBadAccess);
    return;
  }
#endif
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// the warp copies `bytes` (multiple of 16) from src to dst, 16 bytes per lane per step
__device__ __forceinline__ void warp_copy(uint8_t* dst, const uint8_t* src, int bytes, int lane, uint64_t pol) {
  for (int off = lane * 16; off < bytes; off += 512) cp16(dst + off, src + off, pol);
}

// Packed bytes of expert e: computed from the contiguous pool when there is one, so that a task
// start waits on one dependent load (its descriptor) instead of two.
__device__ __forceinline__ const uint8_t* expert_at(const FfnArgs& a, int e) {
  return a.expert_base ? a.expert_base + (size_t)e * a.expert_stride : a.expert_ptr[e];
}

// One unit's descriptor spread over a warp: lane l < 36 holds 32-bit word l (lanes 0..31 only
// hold words 0..31, which cover e, M, pick[8], tok[8], xs[8]; w[8] is words 28..35 and is read
// through a second register).
struct DescRegs {
  int a;  // word lane
  int b;  // word 32 + lane (lanes 0..3)
};
__device__ __forceinline__ DescRegs load_desc(const UnitDesc* U, int lane) {
  const int* w = reinterpret_cast<const int*>(U);
  DescRegs r;
  r.a = __ldg(w + lane);
  r.b = lane < 4 ? __ldg(w + 32 + lane) : 0;
  return r;
}
__device__ __forceinline__ int d_e(const DescRegs& r) { return __shfl_sync(0xffffffffu, r.a, 0); }
__device__ __forceinline__ int d_M(const DescRegs& r) { return __shfl_sync(0xffffffffu, r.a, 1); }
__device__ __forceinline__ int d_pick(const DescRegs& r, int m) { return __shfl_sync(0xffffffffu, r.a, 4 + m); }
__device__ __forceinline__ int d_tok(const DescRegs& r, int m) { return __shfl_sync(0xffffffffu, r.a, 12 + m); }
__device__ __forceinline__ float d_w(const DescRegs& r, int m) {
  // w[m] is word 28 + m: words 28..31 in .a, 32..35 in .b.  Both shuffles run on every lane
  // (a full-mask shuffle must be executed by the whole warp), then each lane selects.
  const int va = __shfl_sync(0xffffffffu, r.a, 28 + (m & 3));
  const int vb = __shfl_sync(0xffffffffu, r.b, m & 3);
  return __int_as_float(m < 4 ? va : vb);
}

// ------------------------------------------------------------------------ gate/up ---
// Each consumer warp streams its own stages (cp.async, `depth` stages ahead) into a private
// ring, so nothing is shared on the data path.  Warp w owns k-tiles kt % 8 == w of every task.
constexpr int kGuRed = 4;                            // partial-sum slots (multiple of kGuEpi)
constexpr int kGuEpi = 2;                            // epilogue warps; task j -> warp j % kGuEpi
constexpr int kGuThreads = (kConsumers + kGuEpi) * 32;
constexpr int kGuTileBytes = 2 * kTileBytes;         // gate tile + up tile of one (row group, k-tile)

struct GuLayout {
  int depth, stage_bytes;
  size_t red_off, ring_off, total;
};

inline GuLayout gu_layout(int mcap, size_t budget) {
  GuLayout L;
  L.stage_bytes = (kGuTileBytes + mcap * 256 + kStageAlign - 1) / kStageAlign * kStageAlign;
  L.red_off = 1024;  // barriers: 2*kGuRed + 1
  L.ring_off = L.red_off + (size_t)kGuRed * kConsumers * 8 * 32 * sizeof(float);
  int depth = (int)((budget - L.ring_off) / ((size_t)kConsumers * L.stage_bytes));
  L.depth = depth > kMaxDepth ? kMaxDepth : depth;
  L.total = L.ring_off + (size_t)kConsumers * L.depth * L.stage_bytes;
  return L;
}

// k-tiles of warp w among the KT k-tiles of one task (kt % 8 == w)
__device__ __forceinline__ int warp_kts(int KT, int w) { return w < KT ? (KT - w + kConsumers - 1) / kConsumers : 0; }

template <int DEPTH, bool ZS>
__global__ void __launch_bounds__(kGuThreads, 2) gateup_kernel(FfnArgs a, GuLayout L) {
  pdl_entry();
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* red_full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* red_empty = red_full + kGuRed;
  uint64_t* never = red_empty + kGuRed;
  float* red = reinterpret_cast<float*>(smem + L.red_off);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* err = a.ws.sync + 1;

#ifdef K3MOE_DEVICE_CHECKS
  if (threadIdx.x == 0) {
    g_chk_err = a.ws.sync + 1;
    g_chk_lo = smem_u32(smem + L.ring_off);
    g_chk_hi = smem_u32(smem + L.total);
  }
  __syncthreads();
#endif
  if (threadIdx.x == 0) {
    for (int i = 0; i < kGuRed; ++i) {
      mbar_init(&red_full[i], kConsumers);
      mbar_init(&red_empty[i], 1);
    }
    mbar_init(never, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  const int RG = a.f / kTileRows;  // row groups of gate/up
  const int KT = a.d / kTileCols;  // k-tiles
  const int ntasks = *a.ws.nunits * RG;
  const size_t gu_stride = (size_t)KT * kGuTileBytes;  // bytes of one row group (gate+up, all k-tiles)
  const int G = gridDim.x;

  if (warp < kConsumers) {
    // ------------------------------------------------------------------ consumers ---
    const int g = lane >> 2, t = lane & 3;
    uint8_t* ring = smem + L.ring_off + (size_t)warp * L.depth * L.stage_bytes;
    const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_normal();
    if (a.test_stall && !wait_phase(never, 0, err, a.wait_ns)) return;
    const int cw = warp_kts(KT, warp);
    const int my_tasks = blockIdx.x < ntasks ? (ntasks - blockIdx.x + G - 1) / G : 0;
    const long long nstages = (long long)my_tasks * cw;

    // issue cursor: task ji, k-tile index ci; descriptors of task ji and ji+1 (prefetched).
    // Wst / x0st: this lane's source bytes of the next stage's weights and of its first token's
    // x fragments; both advance by a constant stride per stage (k-tiles kt, kt+8, ...).
    int ji = 0, ci = 0, Mc = 0;
    DescRegs dcur{0, 0}, dnext{0, 0};
    const uint8_t* Wst = nullptr;
    const uint8_t* x0st = nullptr;
    const uint8_t* xf = reinterpret_cast<const uint8_t*>(a.ws.xfrag);
    const size_t xrow = (size_t)a.d * 2;  // bytes of one token's fragments
    auto enter_task = [&]() {
      Mc = d_M(dcur);
      Wst = expert_at(a, d_e(dcur)) + (size_t)((blockIdx.x + ji * G) % RG) * gu_stride + (size_t)warp * kGuTileBytes +
            lane * 16;
      x0st = xf + (size_t)d_tok(dcur, 0) * xrow + (size_t)warp * 256 + lane * 16;
    };
    if (my_tasks > 0) {
      dcur = load_desc(a.ws.units + blockIdx.x / RG, lane);
      if (my_tasks > 1) dnext = load_desc(a.ws.units + (blockIdx.x + G) / RG, lane);
      enter_task();
    }
    auto issue_next = [&](uint8_t* st) {
      // copy the stage at the issue cursor into `st`, then advance the cursor
      uint8_t* dl = st + lane * 16;
#pragma unroll
      for (int q = 0; q < kGuTileBytes / 512; ++q) cp16(dl + 512 * q, Wst + 512 * q, pol_w);
      if (lane * 16 + 512 * (kGuTileBytes / 512) < kGuTileBytes)
        cp16(dl + 512 * (kGuTileBytes / 512), Wst + 512 * (kGuTileBytes / 512), pol_w);
      if (lane < 16) cp16(dl + kGuTileBytes, x0st, pol_x);
      for (int m = 1; m < Mc; ++m)
        warp_copy(st + kGuTileBytes + m * 256,
                  xf + (size_t)d_tok(dcur, m) * xrow + (size_t)(warp + kConsumers * ci) * 256, 256, lane, pol_x);
      Wst += (size_t)kConsumers * kGuTileBytes;
      x0st += kConsumers * 256;
      if (++ci == cw) {
        ci = 0;
        ++ji;
        dcur = dnext;
        if (ji < my_tasks) enter_task();
        if (ji + 1 < my_tasks) dnext = load_desc(a.ws.units + (blockIdx.x + (ji + 1) * G) / RG, lane);
      }
    };
    // DEPTH groups are always committed ahead (empty ones when there is nothing left to copy),
    // so the stage being consumed is always DEPTH-1 groups behind the newest.
    long long issued = 0;
#pragma unroll
    for (int i = 0; i < DEPTH; ++i) {
      if (issued < nstages) {
        issue_next(ring + (size_t)i * L.stage_bytes);
        ++issued;
      }
      cp_commit();
    }

    int rslot = 0;
    int M_n = my_tasks > 0 ? __ldg(&a.ws.units[blockIdx.x / RG].M) : 0;
    for (int j = 0; j < my_tasks; ++j) {
      const int M = M_n;
      const int gx = g < M ? g : M - 1;
      if (j + 1 < my_tasks) M_n = __ldg(&a.ws.units[(blockIdx.x + (j + 1) * G) / RG].M);
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      for (int c = 0; c < cw; ++c) {
        cp_wait<DEPTH - 1>();
        __syncwarp();
        uint8_t* st = ring + (size_t)rslot * L.stage_bytes;
        uint4 nib[2][2];
        uint2 sc[2];
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          nib[m][0] = lds128(st + m * kTileBytes + lane * 16);
          nib[m][1] = lds128(st + m * kTileBytes + 512 + lane * 16);
          sc[m] = lds64(st + m * kTileBytes + kTileNibBytes + g * 8);
        }
        // lanes of absent tokens (g >= M) read token M-1: the MMA columns they feed are not used
        uint4 xv[4];
#pragma unroll
        for (int b = 0; b < 4; ++b) xv[b] = lds128(st + kGuTileBytes + gx * 256 + (b * 4 + t) * 16);
        __syncwarp();
        if (issued < nstages) {  // refill the slot just read
          issue_next(st);
          ++issued;
        }
        cp_commit();
        rslot = rslot + 1 == DEPTH ? 0 : rslot + 1;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          float bacc[2][4];
#pragma unroll
          for (int st2 = 0; st2 < 2; ++st2) {
            const int w = 2 * (b & 1) + st2;
            const uint32_t b0 = st2 ? xv[b].z : xv[b].x, b1 = st2 ? xv[b].w : xv[b].y;
#pragma unroll
            for (int m = 0; m < 2; ++m) {
              uint32_t A[4];
              dec4(word_of(nib[m][b >> 1], w), A);
              if (st2 == 0)
                mma_zero(bacc[m], A, b0, b1);
              else
                mma_acc(bacc[m], A, b0, b1);
            }
          }
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            const float s_lo = scale_of<ZS>(sc[m].x, b);
            const float s_hi = scale_of<ZS>(sc[m].y, b);
            acc[m][0] = fmaf(bacc[m][0], s_lo, acc[m][0]);
            acc[m][1] = fmaf(bacc[m][1], s_lo, acc[m][1]);
            acc[m][2] = fmaf(bacc[m][2], s_hi, acc[m][2]);
            acc[m][3] = fmaf(bacc[m][3], s_hi, acc[m][3]);
          }
        }
      }
      const int r = j % kGuRed;
      if (j >= kGuRed && !wait_phase(&red_empty[r], (uint32_t)((j / kGuRed - 1) & 1), err, a.wait_ns)) {
        cp_wait<0>();
        return;
      }
      float* rp = red + ((size_t)r * kConsumers + warp) * 8 * 32;
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int q = 0; q < 4; ++q) rp[(m * 4 + q) * 32 + lane] = acc[m][q];
      __syncwarp();
      if (lane == 0) mbar_arrive(&red_full[r]);
    }
    cp_wait<0>();
    return;
  }

  // ------------------------------------------------------------------------ epilogue ---
  {
    const int ew = warp - kConsumers;  // 0..kGuEpi-1: tasks j with j % kGuEpi == ew
    const int g = lane >> 2, t = lane & 3;
    int j = ew;
    int i = blockIdx.x + ew * G;
    // lane m < 8 holds pick m and its x scale of the task's unit; prefetched a task ahead
    int M_n = 0, pick_n = -1;
    float xs_n = 0.f;
    if (i < ntasks) {
      const UnitDesc* U = a.ws.units + i / RG;
      M_n = U->M;
      pick_n = U->pick[lane & 7];
      xs_n = U->xs[lane & 7];
    }
    for (; i < ntasks; i += kGuEpi * G, j += kGuEpi) {
      const int M = M_n, mypick = pick_n;
      const float myxs = xs_n;
      const int inext = i + kGuEpi * G;
      if (inext < ntasks) {
        const UnitDesc* U = a.ws.units + inext / RG;
        M_n = U->M;
        pick_n = U->pick[lane & 7];
        xs_n = U->xs[lane & 7];
      }
      const int r = j % kGuRed;
      if (!wait_phase(&red_full[r], (uint32_t)((j / kGuRed) & 1), err, a.wait_ns)) return;
      float v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float sum = 0.f;
        for (int w = 0; w < kConsumers; ++w) sum += red[(((size_t)r * kConsumers + w) * 8 + q) * 32 + lane];
        v[q] = sum;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&red_empty[r]);

      const int rg = i % RG;
      // SwiGLU for this lane's entries: rows 16rg+g (+8), columns (picks) 2t, 2t+1
      float hmx[2] = {0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int n = 2 * t + c;
        const int p = __shfl_sync(0xffffffffu, mypick, n);
        const float xs = __shfl_sync(0xffffffffu, myxs, n);
        if (n < M) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float gv = v[0 * 4 + 2 * h + c] * xs, uv = v[1 * 4 + 2 * h + c] * xs;
            const float hv = gate_act(gv, a.act) * uv;
            a.ws.hbuf[(size_t)p * a.f + rg * kTileRows + g + 8 * h] = hv;
            hmx[c] = fmaxf(hmx[c], fabsf(hv));
          }
        }
      }
      // max |h| per pick over this task's 16 rows: reduce over the 8 row lanes of each column,
      // then one atomic per (task, pick); hconv_kernel turns it into the pick's fp16 scale
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int n = 2 * t + c;
        const int p = __shfl_sync(0xffffffffu, mypick, n);
        float m = n < M ? hmx[c] : 0.f;
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        if (g == 0 && n < M) atomicMax(a.ws.hmax + p, __float_as_uint(m));
      }
    }
  }
}

// --------------------------------------------------------------------------- hconv ---
// h (fp32, [P][f]) -> fp16 B-fragment rows with one power of two per pick (h = hfrag * hs[p]),
// from the max |h| that gateup_kernel recorded; the max is reset to zero for the next call.
__global__ void __launch_bounds__(128) hconv_kernel(const float* __restrict__ hbuf, uint32_t* hmax, int f, int P,
                                                     __half* __restrict__ hfrag, float* __restrict__ hs) {
  pdl_entry();
  for (int p = blockIdx.x; p < P; p += gridDim.x) {
    const int q = fp16_scale_exp(__uint_as_float(hmax[p]));
    const float inv = exp2i(-q);
    const float* hr = hbuf + (size_t)p * f;
    for (int it = threadIdx.x; it < f / 8; it += blockDim.x) {
      const int blk = it >> 2, tq = it & 3;
      __align__(16) __half h[8];
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        const int kb = 32 * blk + 16 * s2 + 2 * tq;
        h[4 * s2 + 0] = __float2half_rn(hr[kb] * inv);
        h[4 * s2 + 1] = __float2half_rn(hr[kb + 1] * inv);
        h[4 * s2 + 2] = __float2half_rn(hr[kb + 8] * inv);
        h[4 * s2 + 3] = __float2half_rn(hr[kb + 9] * inv);
      }
      *reinterpret_cast<uint4*>(hfrag + (size_t)p * f + (size_t)it * 8) = *reinterpret_cast<const uint4*>(h);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      hs[p] = exp2i(q);
      hmax[p] = 0u;
    }
  }
}

// --------------------------------------------------------------------------- down ---
// Task = (unit, 32 rows of d = two 16-row tile groups) over the whole f range; warp w owns the
// CTA's tasks j % 8 == w and streams each task in chunks of kc k-tiles (one ring stage per chunk:
// kc tiles of each row group, then the unit's h fragments, which both row groups share).
constexpr int kDnThreads = kConsumers * 32;

struct DnLayout {
  int depth, kc, nch, stage_bytes;
  size_t total;
};

inline DnLayout dn_layout(int f, int mcap, size_t budget) {
  DnLayout L;
  const int KT = f / kTileCols;
  const size_t per_kt = 2 * kTileBytes + (size_t)mcap * (4 * 64);  // weights of 2 row groups + h fragments
  int kc = (int)(budget / ((size_t)kConsumers * 2 * per_kt));           // at least 2 stages per warp
  kc = kc < 1 ? 1 : (kc > KT ? KT : kc);
  L.kc = kc;
  L.nch = (KT + kc - 1) / kc;
  L.stage_bytes = (int)((kc * per_kt + kStageAlign - 1) / kStageAlign * kStageAlign);
  int depth = (int)(budget / ((size_t)kConsumers * L.stage_bytes));
  L.depth = depth > kMaxDepth ? kMaxDepth : depth;
  L.total = (size_t)kConsumers * L.depth * L.stage_bytes;
  return L;
}

template <int DEPTH, bool ZS>
__global__ void __launch_bounds__(kDnThreads, 2) down_kernel(FfnArgs a, DnLayout L) {
  pdl_entry();
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  uint32_t* err = a.ws.sync + 1;
  if (a.test_stall) {  // failure-path test: wait on a barrier that nothing completes
    __shared__ uint64_t never;
    if (threadIdx.x == 0) {
      mbar_init(&never, 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (!wait_phase(&never, 0, err, a.wait_ns)) return;
  }

#ifdef K3MOE_DEVICE_CHECKS
  if (threadIdx.x == 0) {
    g_chk_err = a.ws.sync + 1;
    g_chk_lo = smem_u32(smem);
    g_chk_hi = smem_u32(smem + L.total);
  }
  __syncthreads();
#endif
  const int RG2 = a.d / (2 * kTileRows);  // tasks per unit: pairs of 16-row groups
  const int KT = a.f / kTileCols;
  const int ntasks = *a.ws.nunits * RG2;
  const size_t gu_bytes = gateup_region_bytes(a.d, a.f);
  const size_t rg_bytes = (size_t)KT * kTileBytes;  // one row group, all k-tiles
  const int wb = L.kc * kTileBytes;  // weight bytes of one row group's chunk
  const int G = gridDim.x;
  // stage: [kc weight tiles of row group 0][kc of row group 1][M x kc*256 h fragments]
  uint8_t* ring = smem + (size_t)warp * L.depth * L.stage_bytes;
  const uint64_t pol_w = policy_evict_first(), pol_h = policy_evict_normal();
  const int first = blockIdx.x + warp * G, step = kConsumers * G;
  const int my_tasks = first < ntasks ? (ntasks - first + step - 1) / step : 0;
  const long long nstages = (long long)my_tasks * L.nch;

  int ji = 0, ci = 0;
  DescRegs dcur{0, 0}, dnext{0, 0};
  const uint8_t* Wcur = nullptr;  // row group 0 of the task at the issue cursor (row group 1 follows)
  if (my_tasks > 0) {
    dcur = load_desc(a.ws.units + first / RG2, lane);
    if (my_tasks > 1) dnext = load_desc(a.ws.units + (first + step) / RG2, lane);
    Wcur = expert_at(a, d_e(dcur)) + gu_bytes + (size_t)(2 * (first % RG2)) * rg_bytes;
  }
  auto issue_next = [&](uint8_t* st) {
    const int kt0 = ci * L.kc, nk = min(L.kc, KT - kt0);
    warp_copy(st, Wcur + (size_t)kt0 * kTileBytes, nk * kTileBytes, lane, pol_w);
    warp_copy(st + wb, Wcur + rg_bytes + (size_t)kt0 * kTileBytes, nk * kTileBytes, lane, pol_w);
    const int M = d_M(dcur);
    for (int m = 0; m < M; ++m) {
      const int p = d_pick(dcur, m);
      warp_copy(st + 2 * wb + m * L.kc * 256,
                reinterpret_cast<const uint8_t*>(a.ws.hfrag + (size_t)p * a.f) + kt0 * 256, nk * 256, lane, pol_h);
    }
    if (++ci == L.nch) {
      ci = 0;
      ++ji;
      dcur = dnext;
      if (ji < my_tasks)
        Wcur = expert_at(a, d_e(dcur)) + gu_bytes + (size_t)(2 * ((first + ji * step) % RG2)) * rg_bytes;
      if (ji + 1 < my_tasks) dnext = load_desc(a.ws.units + (first + (ji + 1) * step) / RG2, lane);
    }
  };
  // DEPTH groups always committed ahead (see gateup_kernel)
  long long issued = 0;
#pragma unroll
  for (int i = 0; i < DEPTH; ++i) {
    if (issued < nstages) {
      issue_next(ring + (size_t)i * L.stage_bytes);
      ++issued;
    }
    cp_commit();
  }

  int rslot = 0;
  DescRegs dtask = my_tasks > 0 ? load_desc(a.ws.units + first / RG2, lane) : DescRegs{0, 0};
  for (int j = 0; j < my_tasks; ++j) {
    const int i = first + j * step;
    const DescRegs D = dtask;
    if (j + 1 < my_tasks) dtask = load_desc(a.ws.units + (i + step) / RG2, lane);
    const int M = d_M(D);
    const int rg = 2 * (i % RG2);
    // this lane's output columns (picks 2t, 2t+1): pick ids and combine weight x h scale, loaded
    // now so that the epilogue does not wait on them
    int pk[2];
    float osc[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int n = 2 * t + c;
      pk[c] = d_pick(D, n);
      const float wp = d_w(D, n);
      osc[c] = n < M ? wp * __ldg(a.ws.hscale + pk[c]) : 0.f;
    }
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    for (int c = 0; c < L.nch; ++c) {
      cp_wait<DEPTH - 1>();
      __syncwarp();
      uint8_t* st = ring + (size_t)rslot * L.stage_bytes;
      // lanes of absent picks (g >= M) read pick M-1: the MMA columns they feed are not used
      const uint8_t* hrow = st + 2 * wb + (g < M ? g : M - 1) * L.kc * 256;
      const int nk = min(L.kc, KT - c * L.kc);
      for (int kk = 0; kk < nk; ++kk) {
        uint4 u[2][2];
        uint2 sc[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const uint8_t* tp = st + (size_t)r * wb + (size_t)kk * kTileBytes;
          u[r][0] = lds128(tp + lane * 16);
          u[r][1] = lds128(tp + 512 + lane * 16);
          sc[r] = lds64(tp + kTileNibBytes + g * 8);
        }
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const uint4 hv = lds128(hrow + (size_t)(4 * kk + b) * 64 + t * 16);
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const uint4& nv = (b >> 1) ? u[r][1] : u[r][0];
            float bacc[4];
            uint32_t A[4];
            dec4(word_of(nv, 2 * (b & 1)), A);
            mma_zero(bacc, A, hv.x, hv.y);
            dec4(word_of(nv, 2 * (b & 1) + 1), A);
            mma_acc(bacc, A, hv.z, hv.w);
            const float s_lo = scale_of<ZS>(sc[r].x, b);
            const float s_hi = scale_of<ZS>(sc[r].y, b);
            acc[r][0] = fmaf(bacc[0], s_lo, acc[r][0]);
            acc[r][1] = fmaf(bacc[1], s_lo, acc[r][1]);
            acc[r][2] = fmaf(bacc[2], s_hi, acc[r][2]);
            acc[r][3] = fmaf(bacc[3], s_hi, acc[r][3]);
          }
        }
      }
      __syncwarp();
      if (issued < nstages) {
        issue_next(st);
        ++issued;
      }
      cp_commit();
      rslot = rslot + 1 == DEPTH ? 0 : rslot + 1;
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      if (2 * t + c < M) {
        const float sc = osc[c];  // combine weight x the pick's h scale
        float* o = a.ws.obuf + (size_t)pk[c] * a.d + (size_t)rg * kTileRows + g;
        o[0] = acc[0][c] * sc;
        o[8] = acc[0][2 + c] * sc;
        o[kTileRows] = acc[1][c] * sc;
        o[kTileRows + 8] = acc[1][2 + c] * sc;
      }
    }
  }
  cp_wait<0>();
}

// ------------------------------------------------------------------------- combine ---
// y[t][c] = sum over slots 0..k-1, in slot order, of obuf[t*k + slot][c].  A thread owns 4
// columns; its slot loads are issued 8 at a time before any is added.
__global__ void __launch_bounds__(128) combine_kernel(const float* __restrict__ obuf, int T, int d, int k,
                                                       float* __restrict__ y) {
  pdl_entry();
  const size_t n4 = (size_t)T * d / 4;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
    const size_t t = i / (d / 4), c4 = i % (d / 4);
    const float4* src = reinterpret_cast<const float4*>(obuf + (size_t)t * k * d) + c4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < k; s0 += 8) {
      float4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = s0 + j < k ? __ldg(src + (size_t)(s0 + j) * (d / 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (s0 + j < k) {
          acc.x = (s0 + j == 0) ? v[j].x : acc.x + v[j].x;
          acc.y = (s0 + j == 0) ? v[j].y : acc.y + v[j].y;
          acc.z = (s0 + j == 0) ? v[j].z : acc.z + v[j].z;
          acc.w = (s0 + j == 0) ? v[j].w : acc.w + v[j].w;
        }
      }
    }
    reinterpret_cast<float4*>(y)[i] = acc;
  }
}

// two CTAs per SM: 2 x (110 KB + static + 1 KB reserved) fits the SM's 228 KB of shared memory
constexpr int kCtasPerSm = 2;
constexpr size_t kSmemBudget = 110 * 1024;

}  // namespace

namespace {

// Ring depths with an instantiated kernel; the layout's depth is rounded down to one of them.
constexpr int kDepths[] = {2, 3, 4, 6};

template <typename Layout>
int pick_depth(Layout& L, int requested) {
  int d = requested > 0 && requested < L.depth ? requested : L.depth;
  int best = 2;
  for (int v : kDepths)
    if (v <= d) best = v;
  return best;
}

template <int DEPTH, bool ZS>
cudaError_t launch_gu(const FfnArgs& a, const GuLayout& L, cudaStream_t s) {
  static std::atomic<unsigned long long> attr{0};
  const cudaError_t e = set_smem_limit_once(gateup_kernel<DEPTH, ZS>, (int)kSmemBudget, attr);
  if (e != cudaSuccess) return e;
  return launch_pdl(gateup_kernel<DEPTH, ZS>, dim3(a.num_sms * kCtasPerSm), dim3(kGuThreads), L.total, s, a, L);
}

template <int DEPTH, bool ZS>
cudaError_t launch_dn(const FfnArgs& a, const DnLayout& L, cudaStream_t s) {
  static std::atomic<unsigned long long> attr{0};
  const cudaError_t e = set_smem_limit_once(down_kernel<DEPTH, ZS>, (int)kSmemBudget, attr);
  if (e != cudaSuccess) return e;
  return launch_pdl(down_kernel<DEPTH, ZS>, dim3(a.num_sms * kCtasPerSm), dim3(kDnThreads), L.total, s, a, L);
}

}  // namespace

cudaError_t launch_gateup(const FfnArgs& a, cudaStream_t s) {
  const int mcap = a.T < kUnitTokens ? a.T : kUnitTokens;
  GuLayout L = gu_layout(mcap, kSmemBudget);
  L.depth = pick_depth(L, a.ring_depth);
  L.total = L.ring_off + (size_t)kConsumers * L.depth * L.stage_bytes;
  const bool zs = a.zero_scales != 0;
  switch (L.depth) {
    case 2: return zs ? launch_gu<2, true>(a, L, s) : launch_gu<2, false>(a, L, s);
    case 3: return zs ? launch_gu<3, true>(a, L, s) : launch_gu<3, false>(a, L, s);
    case 4: return zs ? launch_gu<4, true>(a, L, s) : launch_gu<4, false>(a, L, s);
    default: return zs ? launch_gu<6, true>(a, L, s) : launch_gu<6, false>(a, L, s);
  }
}

cudaError_t launch_down(const FfnArgs& a, cudaStream_t s) {
  const int mcap = a.T < kUnitTokens ? a.T : kUnitTokens;
  DnLayout L = dn_layout(a.f, mcap, kSmemBudget);
  L.depth = pick_depth(L, a.ring_depth);
  L.total = (size_t)kConsumers * L.depth * L.stage_bytes;
  const bool zs = a.zero_scales != 0;
  switch (L.depth) {
    case 2: return zs ? launch_dn<2, true>(a, L, s) : launch_dn<2, false>(a, L, s);
    case 3: return zs ? launch_dn<3, true>(a, L, s) : launch_dn<3, false>(a, L, s);
    case 4: return zs ? launch_dn<4, true>(a, L, s) : launch_dn<4, false>(a, L, s);
    default: return zs ? launch_dn<6, true>(a, L, s) : launch_dn<6, false>(a, L, s);
  }
}

cudaError_t launch_hconv(const FfnArgs& a, cudaStream_t s) {
  const int P = a.T * a.k;
  return launch_pdl(hconv_kernel, dim3(std::min(P, a.num_sms * 8)), dim3(128), 0, s, (const float*)a.ws.hbuf,
                    a.ws.hmax, a.f, P, a.ws.hfrag, a.ws.hscale);
}

cudaError_t launch_combine(const FfnArgs& a, cudaStream_t s) {
  const size_t n4 = (size_t)a.T * a.d / 4;
  const int grid = (int)std::min<size_t>((n4 + 127) / 128, (size_t)a.num_sms * 16);
  return launch_pdl(combine_kernel, dim3(grid), dim3(128), 0, s, (const float*)a.ws.obuf, a.T, a.d, a.k, a.y);
}

}  // namespace k3
