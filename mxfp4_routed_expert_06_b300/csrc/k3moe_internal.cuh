// k3moe_internal.cuh -- shared definitions of the CUDA path (not part of the C ABI).
#pragma once

#include <atomic>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

#include "../../include/k3moe.h"

namespace k3 {

// ----------------------------------------------------------------------------------------
// Packed MXFP4 layout (the library's own, produced by the pack kernel from the canonical
// layout; lossless).  A matrix of R rows x K columns (R % 16 == 0, K % 128 == 0) is cut into
// tiles of 16 rows x 128 columns, stored tile after tile in (row-group, k-tile) order:
//
//   tile (rg, kt), 1088 bytes:
//     [   0,  512)  unit 0: columns 128kt + [0, 64)     16 bytes per lane L = 4g + t (g < 8, t < 4)
//     [ 512, 1024)  unit 1: columns 128kt + [64, 128)
//     [1024, 1088)  scales: 8 bytes per g: rows (16rg+g) and (16rg+g+8) x 4 blocks of 32 columns,
//                   byte 4*h + b = scale of row 16rg + g + 8h, block b
//   lane L's 16 bytes of unit u: word s (s < 4) holds k16-step s, base column kb = 128kt + 64u + 16s:
//     byte 0: row g,   columns kb+2t, kb+2t+1        byte 1: row g+8, columns kb+2t, kb+2t+1
//     byte 2: row g,   columns kb+2t+8, kb+2t+9      byte 3: row g+8, columns kb+2t+8, kb+2t+9
//     (low nibble = even column), which is exactly the A-operand fragment a0..a7 of
//     mma.m16n8k16 for that k16 step after an e2m1x2 -> f16x2 conversion of each byte.
//
// One expert = [gate/up region][down region]:
//   gate/up: for rg < f/16, kt < d/128: gate tile (rg, kt) then up tile (rg, kt)
//   down:    for rg < d/16, kt < f/128: down tile (rg, kt)
// Total bytes = 3*f*d/2 + 3*f*d/32, the canonical count.
// ----------------------------------------------------------------------------------------
constexpr int kTileRows = 16;
constexpr int kTileCols = 128;
constexpr int kTileBytes = 1088;
constexpr int kTileNibBytes = 1024;

__host__ __device__ inline size_t packed_expert_bytes(int d, int f) { return 3ull * (size_t)f * d / 2 + 3ull * (size_t)f * d / 32; }
__host__ __device__ inline size_t gateup_region_bytes(int d, int f) { return (size_t)(f / 16) * (d / 128) * 2 * kTileBytes; }

// B-operand fragments of the activations (fp16), for one row of K values (x: K = d, h: K = f):
//   frag[row][blk][t][16 bytes], blk < K/32, t < 4; the 16 bytes hold, for the two k16 steps of
//   block blk (kb = 32 blk + 16 s, s = 0, 1), the halves (kb+2t, kb+2t+1, kb+2t+8, kb+2t+9):
//   i.e. registers b0b1, b2b3 of step 0 then of step 1, as mma.m16n8k16 expects for column n.
// Row stride = K * 2 bytes.

// A work unit is (expert, up to kUnitTokens consecutive picks of that expert): the FFN kernels
// multiply one unit's tokens as the n = 8 columns of mma.m16n8k16.  Bucketing writes one flat
// descriptor per unit so that the FFN kernels fetch everything about a unit in one go.
constexpr int kUnitTokens = 8;
struct __align__(16) UnitDesc {
  int e;                    // expert id
  int M;                    // picks in the unit (1..8)
  int pbase;                // index of the unit's first pick in perm
  int pad;
  int pick[kUnitTokens];    // pick ids p = t*k + slot
  int tok[kUnitTokens];     // token ids t
  float xs[kUnitTokens];    // power-of-two scale of the token's fp16 image
  float w[kUnitTokens];     // combine weight of the pick
};
static_assert(sizeof(UnitDesc) == 144, "UnitDesc is 9 x 16 bytes");

// Workspace of one layer, sized for T_max tokens (P = T_max*k picks).
struct Workspace {
  float* logits = nullptr;      // [T_max][E]
  __half* xfrag = nullptr;      // [T_max][d] fragment order
  float* xscale = nullptr;      // [T_max] power of two: x = xfrag * xscale
  int32_t* idx = nullptr;       // [T_max][k]
  float* w = nullptr;           // [T_max][k]
  int32_t* counts = nullptr;    // [E]
  int32_t* offsets = nullptr;   // [E+1]
  int32_t* perm = nullptr;      // [P]
  int32_t* act = nullptr;       // [E] active experts in id order
  int32_t* nact = nullptr;      // [1]
  UnitDesc* units = nullptr;    // [P/8 + E] work units
  int32_t* nunits = nullptr;    // [1]
  float* hbuf = nullptr;        // [P][f] SwiGLU output, fp32
  __half* hfrag = nullptr;      // [P][f] fragment order
  float* hscale = nullptr;      // [P] power of two per pick (h = hfrag * hscale)
  float* obuf = nullptr;        // [P][d] w-scaled expert outputs
  uint32_t* sync = nullptr;     // [16]: [0] router last-block ticket, [1] device error flags
  int32_t* bad = nullptr;       // [4] pack time: [0] error flags, [1] min scale byte, [2] max scale byte
  // tensor-core path (large T); it also reuses obuf (first as xg, the fp16 rows of x in bucketed
  // order [P][d], which the down projection then overwrites), hbuf (fp32 h [P][f]), hfrag (as
  // h16 [P][f]) and hscale (as the per-row power of two of h16), xscale (per-token power of two)
  uint32_t* hmax = nullptr;     // [P] float bits of max |h| (per pick on the decode path, per bucketed
                                //     row on the GEMM path); zero between calls
  int4* mtiles = nullptr;       // [P/128 + E] {expert, first bucketed row, rows, 0}
  int32_t* nmtiles = nullptr;   // [1]
  int32_t* chist = nullptr;     // [P/2048 + 1][E] per-chunk expert counts (multi-CTA bucketing)
};

enum KernelId {
  KID_ROUTER = K3MOE_K_ROUTER,
  KID_TOPK = K3MOE_K_TOPK,
  KID_BUCKET = K3MOE_K_BUCKET,
  KID_GATEUP = K3MOE_K_GATEUP,
  KID_DOWN = K3MOE_K_DOWN,
  KID_GEMM_GU = K3MOE_K_GEMM_GU,
  KID_GEMM_DN = K3MOE_K_GEMM_DN,
  KID_COMBINE = K3MOE_K_COMBINE,
  KID_GATHER = K3MOE_K_GATHER,
};

// Kernel launchers (defined in the .cu files).  All return cudaGetLastError().
struct RouterArgs {
  const uint16_t* x;      // [T][d] bf16
  const float* Wr;        // [E][d]
  const float* bias;      // [E] or nullptr
  int T, d, E, k;
  Workspace ws;
  int fuse_select;        // 1: last block also does top-k + bucketing (small T)
  int need_counts;        // 1: the fused bucketing also writes counts / offsets (tensor-core FFN follows)
};
cudaError_t launch_router(const RouterArgs& a, cudaStream_t s);
cudaError_t launch_convert(const RouterArgs& a, int num_sms, cudaStream_t s);  // x -> xfrag, xscale
cudaError_t launch_topk(const float* logits, const float* bias, int T, int E, int k, int32_t* idx, float* w,
                        cudaStream_t s);
cudaError_t launch_bucket(const int32_t* idx, int T, int k, int E, int32_t* counts, int32_t* offsets,
                          int32_t* perm, int32_t* act, int32_t* nact, UnitDesc* units, int32_t* nunits,
                          const float* w, const float* xscale, int32_t* chist, cudaStream_t s,
                          bool fill_units = true);

// Atomic add with acquire-release semantics at GPU scope: the caller's earlier writes (and those
// it observed through a barrier) are visible to whoever reads the new value, and the caller
// sees the writes that preceded the earlier adds.
__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Programmatic dependent launch.  Every kernel of the forward path begins with pdl_entry(): it
// waits until the previous kernel in the stream has completed and its writes are visible, then
// lets the next kernel be scheduled.  Only launch latency and CTA start-up overlap; no kernel
// touches global memory before its predecessor has finished.
__device__ __forceinline__ void pdl_entry() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

// Raises a kernel's dynamic shared-memory limit on the current device.  The attribute belongs
// to the device, so each call site keeps one bit per device (devices 0..63) and sets it the
// first time that device launches the kernel; a process that drives several GPUs sets it on
// each of them.  Devices beyond 63 set it on every call.
template <typename Fn>
inline cudaError_t set_smem_limit_once(Fn* kernel, int bytes, std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit != 0ull && (done.load(std::memory_order_acquire) & bit) != 0ull) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit != 0ull) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Gate activation of the expert FFN, h = gate_act(g) * u (K3MOE_ACT_*).  SwiGLU keeps the exact
// expression silu(g) = g / (1 + exp(-g)); SiTU-GLU is beta1 * beta2 * sigmoid(g) * tanh(g / beta2)
// with beta1 = 4, beta2 = 25 (the pages' parameters; the formula is a reading of their glossary).
constexpr float kSituBeta1 = 4.0f, kSituBeta2 = 25.0f;
__device__ __forceinline__ float gate_act(float g, int act) {
  if (act == K3MOE_ACT_SITU_GLU) return kSituBeta1 * kSituBeta2 * (1.0f / (1.0f + expf(-g))) * tanhf(g / kSituBeta2);
  return g / (1.0f + expf(-g));
}

// Device error flags (ws.sync[1]).
constexpr uint32_t kErrTimeout = 1u;
constexpr uint32_t kErrBadAccess = 2u;  // self-checking builds only: a copy address failed its check
constexpr uint32_t kErrBudget = 4u;     // device-side cache lookup: a call needed more experts than slots

struct FfnArgs {
  const uint8_t* const* expert_ptr;  // [E] device pointers to each expert's packed block
  int d, f, E, k, T;
  Workspace ws;
  float* y;                          // [T][d]
  int num_sms;                       // persistent grid size
  unsigned long long wait_ns;        // bound on every device-side wait
  int test_stall;                    // 1: consumers wait on a barrier nothing arrives at (timeout test)
  int ring_depth;                    // 0: automatic; else stages in flight per streaming warp
  int zero_scales;                   // 1: some E8M0 scale byte is 0 (exact subnormal decode needed)
  const uint8_t* expert_base;        // non-null: expert e is at expert_base + e * expert_stride (no
  size_t expert_stride;              //   table lookup); null: expert_ptr[e] (device cache mode)
  int act;                           // gate activation (K3MOE_ACT_*)
};
cudaError_t launch_gateup(const FfnArgs& a, cudaStream_t s);
cudaError_t launch_down(const FfnArgs& a, cudaStream_t s);
cudaError_t launch_hconv(const FfnArgs& a, cudaStream_t s);
cudaError_t launch_combine(const FfnArgs& a, cudaStream_t s);
// Tensor-core grouped GEMM path (gemm_tc.cu).
struct GemmFfn {
  const uint8_t* const* expert_ptr;
  int d, f, k, T;
  int s_ref;                 // weights enter fp16 as e2m1 * 2^(s - s_ref)
  float wscale;              // 2^(s_ref - 127)
  const int4* mtiles;
  const int32_t* nmtiles;
  const int32_t* perm;
  const float* w;            // [P] combine weights by pick
  float* xs;                 // [T] power of two per token
  __half* xg;                // [P][d] fp16 image of x, rows in bucketed order
  float* hbuf;               // [P][f]
  uint32_t* hmax;            // [P]
  __half* h16;               // [P][f]
  float* hs;                 // [P]
  float* obuf;               // [P][d]
  uint32_t* err;
  unsigned long long wait_ns;
  int num_sms;
  int act;                   // gate activation (K3MOE_ACT_*)
};
bool gemm_scales_ok(int s_min, int s_max);
cudaError_t launch_gemm_prep(const GemmFfn& q, const uint16_t* x, const int32_t* counts, const int32_t* offsets,
                             int E, cudaStream_t s);
cudaError_t launch_gemm_gu(const GemmFfn& q, cudaStream_t s);
cudaError_t launch_gemm_h16(const GemmFfn& q, int P, cudaStream_t s);
cudaError_t launch_gemm_dn(const GemmFfn& q, cudaStream_t s);
// router logits on the tensor cores for large T: x (bf16 [T][d], 16-byte aligned) against W_r
// split into bf16 hi and lo halves (wsplit [E][2d]) -> logits fp32 [T][E]
cudaError_t launch_router_tc(const uint16_t* x, int T, int d, int E, const uint16_t* wsplit, float* logits,
                             uint32_t* err, unsigned long long wait_ns, int num_sms, cudaStream_t s);
cudaError_t launch_split_router(const float* W, int E, int d, uint16_t* out, cudaStream_t s);
cudaError_t launch_residual_rmsnorm(const float* y, const uint16_t* x, int T, int d, float eps, uint16_t* x_next,
                                    uint16_t* x_norm, cudaStream_t s);

// Zero-copy miss path of the expert cache: copy n experts of `bytes` each from the mapped pinned
// pool (device view) into their slots, in one launch on `s`.
struct MissCopy {
  const uint8_t* src;  // device address of the expert in the mapped pinned pool
  uint8_t* dst;        // its device slot
};
cudaError_t launch_miss_copy(const MissCopy* list, int n, size_t bytes, int num_sms, cudaStream_t s);

// Device-side LRU of the expert cache (k3moe_cache_set_device_lru).
struct LruState {
  int head, tail;                                  // most / least recently used slot (-1: none)
  unsigned long long hits, misses, evictions, calls;
};
struct LruArgs {
  LruState* state;
  int32_t* prev;            // [n_slots] LRU list links
  int32_t* next;
  int32_t** owner;          // [n_slots] the layer's slot_of entry that holds the slot, or null
  int n_slots;
  uint8_t* slots;           // slot s at slots + s * slot_bytes
  size_t slot_bytes;
  const int32_t* act;       // [nact] active experts of the call, ascending
  const int32_t* nact;
  int32_t* slot_of;         // [E] the layer's expert -> slot (-1: not resident)
  const uint8_t** eptr;     // [E] device pointer table the FFN kernels read
  const uint8_t* pool_dev;  // the layer's mapped pinned pool
  MissCopy* miss;           // [E] out: the call's misses
  int32_t* nmiss;           // out: their count
  uint32_t* err;            // device error flags
};
cudaError_t launch_lru_lookup(const LruArgs& a, cudaStream_t s);
cudaError_t launch_miss_copy_dev(const MissCopy* list, const int32_t* n_dev, int max_n, size_t bytes, int num_sms,
                                 cudaStream_t s);
cudaError_t launch_lru_detach(LruState* st, int32_t* prev, int32_t* next, int32_t** owner, int n_slots,
                              const int32_t* slot_of, int E, cudaStream_t s);

// canon_nib/canon_scl point at the canonical bytes of the first of n_exp experts; dst at its packed block.
cudaError_t launch_pack(const uint8_t* canon_nib, const uint8_t* canon_scl, int n_exp, int d, int f, uint8_t* dst,
                        int32_t* bad, cudaStream_t s);

// Sets the message k3moe_last_error() returns on this thread.
void set_last_error(const char* msg);

// p is a multiple of n bytes (n a power of two).  The kernels access caller buffers with their
// natural (or vector) width and a misaligned access is a device fault, so the entry points refuse
// such pointers before any work is queued.
inline bool aligned_to(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; }

}  // namespace k3
