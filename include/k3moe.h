/*
 * k3moe.h -- C ABI of the routed mixture-of-experts layer on MXFP4 experts (B300, sm_103a).
 *
 * The layer (pages on the kimi-k3-in-c engine, fiv.co.kr "kimi-k3-in-c deep dive"):
 *   router      sigmoid scores of x against W_r; a per-expert bias steers the selection
 *               only; the top-k experts (16 of 896 in Kimi K3) are mixed with weights taken
 *               from the unbiased scores, renormalised to sum 1
 *               (section "what you learn", router paragraph; invariants table, row 5;
 *               glossary entry MoE)
 *   experts     every expert is a SwiGLU FFN whose gate/up/down weights stay MXFP4 -- E2M1
 *               nibbles with one E8M0 scale per 32 values, value = E2M1[nibble]*2^(scale-127)
 *               -- and are multiplied without being expanded to a dense copy
 *               (section "four reductions", reduction 1; glossary entry MXFP4)
 *   combine     y[t] = sum over the k slots, in slot order, of w[t,slot] * expert_out
 *   cache       an LRU expert cache whose size changes speed, never the output
 *               (section "four reductions", expert LRU paragraph; opening: "the output is
 *               byte-identical whatever the memory budget")
 *
 * Conventions for every call:
 *   - Return 0 on success or a negative K3MOE_ERR_* code; k3moe_last_error() then gives a
 *     message (thread-local, valid until the next failing call on the same thread).
 *   - Arguments are checked before any device work is queued; a failed check changes nothing.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  Device
 *     work is queued on it asynchronously unless a call says otherwise.
 *   - "device pointer" means memory of the current CUDA device, allocated by the caller (for
 *     example by PyTorch); the library never frees caller memory.  The library owns what it
 *     allocates: packed weights, workspace, cache slots, pinned pools.
 *   - One layer object must not be used from two streams at the same time: calls share its
 *     workspace.  Different layer objects are independent (a shared cache excepted).
 *   - Device buffers are aligned at least to their element size (int32 and float32: 4 bytes,
 *     bf16: 2 bytes); x of the router and of the layer forward, and y of the layer forward, to
 *     16 bytes.  A misaligned device pointer is refused with INVALID_ARG (a misaligned access
 *     would be a device fault).  Host buffers of the host-buffer entry point need no alignment.
 *   - Canonical MXFP4 input layout, per expert e (experts back to back):
 *       nibbles  [3][rows][cols/2] bytes: matrix 0 = gate W_g [f][d], 1 = up W_u [f][d],
 *                2 = down W_d [d][f]; element 2i of a row in the LOW nibble of byte i;
 *                E2M1 codes per OCP MX v1.0 (bit 3 sign, bits 2..1 exponent, bit 0 mantissa)
 *       scales   [3][rows][cols/32] E8M0 bytes; block b of a row covers columns 32b..32b+31
 *     so one expert is 3*f*d/2 nibble bytes + 3*f*d/32 scale bytes (17,547,264 bytes in total
 *     at d=7168, f=1536, the count printed in "four reductions", reduction 1).
 */
#ifndef K3MOE_H
#define K3MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define K3MOE_OK 0
#define K3MOE_ERR_INVALID_ARG (-1)      /* bad pointer, size, dimension or option */
#define K3MOE_ERR_OOM (-2)              /* device or pinned host allocation failed */
#define K3MOE_ERR_CUDA (-3)             /* a CUDA runtime call or kernel launch failed */
#define K3MOE_ERR_TIMEOUT (-4)          /* a bounded device-side wait gave up */
#define K3MOE_ERR_BUDGET_TOO_SMALL (-5) /* the cache cannot hold the experts one call needs */
#define K3MOE_ERR_UNSUPPORTED (-6)      /* a valid request the library does not serve */

/* Layer dimensions, validated strictly (unknown or inconsistent values are refused, never
 * defaulted -- the engine's strict config loading, "what you learn", last paragraph):
 *   d      model width, multiple of 128, <= 16384
 *   f      expert intermediate width, multiple of 128, <= 16384
 *   E      number of routed experts, 1..4096
 *   k      experts per token, 1..min(E, 32)
 *   T_max  largest token count a call may pass, 1..65536 (sizes the workspace) */
typedef struct {
  int d, f, E, k, T_max;
} k3moe_dims;

typedef struct k3moe_layer k3moe_layer; /* opaque: packed weights, router, workspace */
typedef struct k3moe_cache k3moe_cache; /* opaque: device expert slots + LRU state */

typedef struct {
  uint64_t hits;       /* experts found resident */
  uint64_t misses;     /* experts copied from the pinned pool */
  uint64_t evictions;  /* resident experts replaced */
  uint64_t h2d_bytes;  /* bytes copied host -> device (misses and prefetches) */
  double h2d_ms;       /* device time of those copies (CUDA events on the copy stream) */
  uint64_t calls;      /* layer calls served */
  uint64_t prefetched; /* experts copied by k3moe_cache_prefetch (their bytes are in h2d_bytes and
                          their copy time in h2d_ms; a later call that finds one counts a hit) */
} k3moe_cache_stats_t;

/* Bytes of one expert in the packed device layout (equal to the canonical byte count:
 * 3*f*d/2 + 3*f*d/32).  Returns 0 for invalid dims. */
size_t k3moe_packed_expert_bytes(const k3moe_dims* dims);

/* Build a layer: repack all E experts from the canonical layout into the library's packed
 * layout (16-row x 128-column tiles, nibbles in tensor-core fragment order with each tile's
 * scales stored right after it; lossless), and copy the router.
 *   dims          layer dimensions (see k3moe_dims)
 *   canon_nib     E * 3*f*d/2 bytes, canonical nibbles of experts 0..E-1
 *   canon_scale   E * 3*f*d/32 bytes, canonical E8M0 scales; a scale byte of 255 (NaN) is
 *                 refused with K3MOE_ERR_INVALID_ARG (checked on the device, reported here)
 *   src_on_device 1: canon_nib, canon_scale, W_r and bias are device pointers; 0: host
 *   W_r           router weights [E][d] float32, row-major
 *   bias          selection bias [E] float32, or NULL for all zeros
 *   cache         NULL: packed experts live in device memory owned by the layer.
 *                 non-NULL: they live in a pinned host pool owned by the layer, and are
 *                 brought to the device through `cache` (which may serve several layers)
 *   stream        stream for the copies and the pack kernel; the call synchronises it
 *                 before returning (the source buffers may be freed afterwards)
 *   out           receives the new layer; free it with k3moe_layer_free
 * Errors: INVALID_ARG (dims, NULL pointers, NaN scale), OOM, CUDA. */
int k3moe_pack_experts(const k3moe_dims* dims, const void* canon_nib, const void* canon_scale, int src_on_device,
                       const float* W_r, const float* bias, k3moe_cache* cache, void* stream, k3moe_layer** out);

/* Packed-pool header.  It describes a packed expert pool (the bytes k3moe_read_packed returns,
 * experts 0..E-1 back to back) so that a saved pool can be validated and loaded again with
 * k3moe_layer_from_packed, without repacking from the canonical layout.  The pages' engine
 * streams a prepacked trunk ("one layer = one read"); this is the expert-pool counterpart. */
#define K3MOE_POOL_MAGIC 0x584D334Bu /* the bytes "K3MX" */
#define K3MOE_POOL_VERSION 1         /* the 16 x 128 tile layout this library writes */
typedef struct {
  uint32_t magic;         /* K3MOE_POOL_MAGIC */
  uint32_t version;       /* K3MOE_POOL_VERSION */
  int32_t d, f, E;        /* dimensions of the experts and their count */
  int32_t s_min, s_max;   /* smallest and largest E8M0 scale byte in the pool */
  int32_t zero_scales;    /* 1 when some scale byte is 0 (then s_min is 0) */
  uint64_t expert_bytes;  /* packed bytes per expert (k3moe_packed_expert_bytes) */
  uint64_t checksum;      /* FNV-1a 64 of every byte of the header before this field */
} k3moe_pool_header;

/* Fill `out` for the layer's packed pool.  Errors: INVALID_ARG (NULL). */
int k3moe_pool_header_get(k3moe_layer* layer, k3moe_pool_header* out);
/* 0 when `header` describes a pool this library can load for `dims` (magic, version, checksum,
 * d, f, E, expert size, a valid scale range), else INVALID_ARG with the mismatch in the message.
 * Host only. */
int k3moe_pool_header_check(const k3moe_pool_header* header, const k3moe_dims* dims);
/* Build a layer from a packed pool (as saved from k3moe_read_packed, with its header) instead of
 * canonical bytes; otherwise as k3moe_pack_experts (router, bias, cache and stream arguments, and
 * ownership).  packed: E * header->expert_bytes bytes, host or device per src_on_device.  The pool
 * is copied as is (it is trusted to match the header; the header is checked first).  Errors:
 * INVALID_ARG (a header that fails k3moe_pool_header_check, NULL pointers), OOM, CUDA. */
int k3moe_layer_from_packed(const k3moe_dims* dims, const k3moe_pool_header* header, const void* packed,
                            int src_on_device, const float* W_r, const float* bias, k3moe_cache* cache, void* stream,
                            k3moe_layer** out);

/* Router alone ("what you learn", router paragraph; invariants row 5):
 *   logit[t,e] = sum_j x[t,j]*W_r[e,j] (fp32 accumulate), sigma = 1/(1+exp(-logit)),
 *   key = sigma + bias[e]; idx[t,:] = the k experts with the largest keys in descending key
 *   order, ties to the lower expert id; w[t,i] = sigma[idx[t,i]] / sum_i sigma[idx[t,i]].
 * From 64 tokens the logits run on the tensor cores with W_r split into bf16 hi + lo parts
 * (each weight to 2^-18 relative), at most 4e-4 from the fp32 sum: keys closer than that may
 * rank differently than with the CUDA-core sum used below 64 tokens.
 *   x    device pointer, [T][d] bf16, row-major, 16-byte aligned
 *   T    1..T_max
 *   idx  device pointer, [T][k] int32 (output)
 *   w    device pointer, [T][k] float32 (output)
 * Errors: INVALID_ARG, CUDA. */
int k3moe_router_topk(k3moe_layer* layer, const void* x_bf16, int T, int32_t* idx, float* w, void* stream);

/* Router + top-k without any device allocation, and without a layer object.  The pages
 * have no counterpart: this entry point exists for callers that cannot call cudaMalloc --
 * code running inside a host framework whose memory pool already owns the device memory
 * (another allocation may fail or bypass the framework's accounting), or loops where an
 * allocation's implicit device synchronisation is not acceptable.  It applies the same routing
 * rule as k3moe_router_topk, with the same ranking (descending sigma + bias, ties to the lower
 * expert id, NaN and infinite keys ordered by their bits, every id in 0..E-1), but its fp32
 * logits come from its own GEMV, whose summation order differs from k3moe_router_topk's (and
 * from 64 tokens on, k3moe_router_topk computes the logits on the tensor cores from W_r split
 * into bf16 hi + lo, within 4e-4 of fp32).  So: idx equals k3moe_router_topk's on every token
 * whose k-th and (k+1)-th keys differ by at least 1e-3, and w agrees within 1e-5.  It reads
 * caller buffers:
 *   x     device, [T][d] bf16 (8-byte aligned);  W_r device, [E][d] float32 (16-byte aligned)
 *   bias  device, [E] float32, or NULL;  idx device, [T][k] int32;  w device, [T][k] float32
 *   d multiple of 4; 1 <= E <= 4096; 1 <= k <= min(E, 32); T*E <= 65536 (larger requests are
 *   refused with K3MOE_ERR_INVALID_ARG).
 * Its scratch (the T*E router logits and a block-election ticket) is one fixed 256 KiB + 256 B
 * array in the library's device memory, held by every GPU that loads the library until the
 * process exits.  The first call on a device does a one-time set-up with that device current
 * (it looks up the array's device address); make that first call before any stream capture.
 * Every call on a device shares the array, which keeps the previous call's contents; the
 * ticket is cleared on `stream` before each launch.  Calls that overlap on the GPU (on two
 * streams at once) race on the array and give undefined results.
 * Errors: INVALID_ARG, CUDA. */
int k3moe_router_topk_noalloc(const void* x_bf16, const float* W_r, const float* bias, int T, int d, int E, int k,
                              int32_t* idx, float* w, void* stream);

/* Token-to-expert bucketing of T*k picks (pick p = t*k + slot):
 *   counts[e]  number of picks routed to expert e                      [E] int32
 *   offsets    exclusive prefix sum of counts in expert-id order       [E+1] int32
 *   perm       for each expert in id order, its picks in ascending p   [T*k] int32
 * Deterministic (a pure function of idx).  All pointers are device pointers.
 *   idx  [T][k] int32 expert ids, each in 0..E-1 (ids out of range: the pick is dropped from
 *        every expert and perm's tail is left unspecified; no memory outside the outputs is
 *        touched).
 * Errors: INVALID_ARG, CUDA. */
int k3moe_bucket(k3moe_layer* layer, const int32_t* idx, int T, int32_t* counts, int32_t* offsets, int32_t* perm,
                 void* stream);

/* The whole layer: router -> top-k -> bucketing -> per-expert SwiGLU FFN on the MXFP4
 * weights -> combine ("four reductions", reduction 1; invariants row 5):
 *   y[t,:] = sum_{slot=0..k-1} w[t,slot] * W_d,e (silu(W_g,e x_t) * (W_u,e x_t)),
 *   e = idx[t,slot], silu(z) = z/(1+exp(-z)), summed in slot order (K3MOE_OPT_ACTIVATION
 *   selects SiTU-GLU instead of silu).
 *   x  device pointer, [T][d] bf16 row-major, 16-byte aligned;
 *   y  device pointer, [T][d] float32 (output), 16-byte aligned.
 *   T  1..T_max.  y excludes any residual.
 * The result does not depend on the cache budget, on which experts were resident, or on
 * the run (bitwise).  Small T runs the register-decode path, large T the tcgen05 grouped
 * GEMM path (k3moe_set_option); the two agree within the accuracy bound, not bitwise.
 * In cache mode the call synchronises `stream` once (to learn which experts it needs), unless
 * every expert of the layer already sits in a slot and the cache has a slot for every expert
 * of every layer using it (then nothing can be evicted and the lookup is skipped), or the cache
 * keeps its LRU state on the device (k3moe_cache_set_device_lru: no host round trip).
 * A device-resident layer's call only queues work on `stream` (no host synchronisation, no
 * allocation), so it can be captured into a CUDA graph by stream capture and replayed with the
 * same bytes, after one eager call of each path has run (that call sets the kernels' attributes);
 * capture with per-kernel timing (k3moe_profile) off.
 * Errors: INVALID_ARG, CUDA, TIMEOUT, BUDGET_TOO_SMALL, OOM (cache mode). */
int k3moe_layer_forward(k3moe_layer* layer, const void* x_bf16, int T, float* y, void* stream);

/* k3moe_layer_forward with HOST buffers: copies x (host, [T][d] bf16) to the device, runs
 * the layer, copies y back to host ([T][d] float32) and synchronises `stream`.  Pinned host
 * memory gives the fastest copies; pageable memory also works; neither needs any alignment
 * (device staging buffers hold x and y).  Errors as layer_forward. */
int k3moe_layer_forward_host(k3moe_layer* layer, const void* x_bf16_host, int T, float* y_host, void* stream);

/* Repeated layer calls as one CUDA graph (a decode loop's launch overhead leaves the host).
 * k3moe_graph_create runs `calls` layer calls of T tokens once, eagerly on `stream` (call c reads
 * x + c*T*d bf16 values and writes y + c*T*d floats, as k3moe_layer_forward does; the eager run
 * also sets the kernels' launch attributes), then captures the same calls on a private stream
 * into a graph.  k3moe_graph_launch replays them on `stream` with the same bytes; inputs are read
 * and outputs written at the addresses given at creation.  k3moe_sync reports device-side
 * failures of replayed calls as of eager ones.
 *   layer   device-resident (packed without a cache: cache-mode calls synchronise the host),
 *           per-kernel timing (k3moe_profile) off
 *   x, y    device pointers, 16-byte aligned, [calls*T][d] bf16 and [calls*T][d] float32
 *   T       1..T_max;  calls >= 1
 * The graph holds the layer's workspace: replays of graphs of one layer, and its other calls,
 * must be ordered (one stream).  It replays the calls as captured: options set later (path,
 * activation, wait bound) do not reach it; create a new graph for them.  Destroy it before the
 * layer.
 * Errors: INVALID_ARG, UNSUPPORTED (cache mode), CUDA, OOM, and those of k3moe_layer_forward. */
typedef struct k3moe_graph k3moe_graph;
int k3moe_graph_create(k3moe_layer* layer, const void* x_bf16, int T, int calls, float* y, void* stream,
                       k3moe_graph** out);
int k3moe_graph_launch(k3moe_graph* graph, void* stream);
void k3moe_graph_destroy(k3moe_graph* graph);

/* Synchronise the layer's last stream and report device-side failures: every wait inside
 * the kernels is bounded (K3MOE_OPT_DEVICE_WAIT_NS, default 2 s); a wait that gives up sets a
 * device flag and its kernel returns early.  This call returns K3MOE_ERR_TIMEOUT (and clears the
 * flag) if that happened since the previous check; the outputs of those calls are invalid.
 * k3moe_layer_forward_host does the same check itself. */
int k3moe_sync(k3moe_layer* layer);

/* Options. */
#define K3MOE_OPT_PATH 1        /* value: K3MOE_PATH_AUTO (default), _DECODE, _GEMM */
#define K3MOE_OPT_GEMM_MIN_T 2  /* value: smallest T the AUTO path sends to the grouped GEMM
                                   (default 512; layers whose scale bytes span more than 36
                                   steps always take the register-decode path under AUTO) */
#define K3MOE_OPT_DEVICE_WAIT_NS 3  /* value: bound in ns on every device-side wait (1e6..6e10) */
#define K3MOE_OPT_TEST_STALL 4  /* value 1: the next forward's FFN kernels wait on a barrier that
                                   nothing completes until the bound expires (failure-path test) */
#define K3MOE_OPT_RING_DEPTH 5  /* value 0 (default): automatic; 1..6: stages each streaming warp
                                   keeps in flight (a tuning and test knob; results do not change) */
#define K3MOE_OPT_TEST_FAIL_COPY 7  /* value n > 0: the n-th cache copy from now (a miss, or a
                                   prefetch) reports a failure without copying (failure-path test).
                                   That call returns K3MOE_ERR_CUDA; the slot it was filling is
                                   forgotten, so later calls copy the expert again and their
                                   results are unchanged */
#define K3MOE_OPT_ACTIVATION 8   /* value: K3MOE_ACT_SWIGLU (default) or K3MOE_ACT_SITU_GLU */
#define K3MOE_OPT_MISS_PATH 9    /* cache mode: how a call's missed experts reach their slots.
                                    K3MOE_MISS_COPY_ENGINE (default): one cudaMemcpyAsync per miss
                                    on the cache's copy stream.  K3MOE_MISS_ZERO_COPY: one kernel on
                                    the layer's stream copies every miss of the call, the SMs
                                    reading the mapped pinned pool directly.  The output does not
                                    depend on the choice (the FFN reads the slots either way) */
#define K3MOE_MISS_COPY_ENGINE 0
#define K3MOE_MISS_ZERO_COPY 1
#define K3MOE_PATH_AUTO 0
#define K3MOE_PATH_DECODE 1
#define K3MOE_PATH_GEMM 2
/* Gate activations (h = act(g) * u in every expert):
 *   K3MOE_ACT_SWIGLU    act(g) = silu(g) = g / (1 + exp(-g)), the activation the layer specification names
 *   K3MOE_ACT_SITU_GLU  act(g) = beta1 * beta2 * sigmoid(g) * tanh(g / beta2), beta1 = 4, beta2 = 25.
 *                       The kimi-k3-in-c deep dive (glossary entry SiTU-GLU) names K3's activation as a
 *                       tanh-sigmoid combination whose beta1 = 4 and beta2 = 25 bound the gate above by
 *                       100; it prints no formula, so this one is a reading: it is bounded by
 *                       beta1 * beta2 = 100, tends to 0 as g -> -inf and has slope beta1 / 2 at 0. */
#define K3MOE_ACT_SWIGLU 0
#define K3MOE_ACT_SITU_GLU 1
int k3moe_set_option(k3moe_layer* layer, int option, long long value);

/* Per-kernel device times (CUDA events around each launch, on the launch stream).
 * k3moe_profile(layer, 1) clears the totals and starts recording; (layer, 0) stops.
 * k3moe_profile_read synchronises the layer's last stream and fills `out` (K3MOE_K_COUNT
 * entries). */
enum {
  K3MOE_K_ROUTER = 0,   /* router logits (+ fused top-k and bucketing for small T) */
  K3MOE_K_TOPK = 1,     /* top-k for large T */
  K3MOE_K_BUCKET = 2,   /* bucketing for large T */
  K3MOE_K_GATEUP = 3,   /* gate/up + SwiGLU, register-decode path */
  K3MOE_K_DOWN = 4,     /* down projection, register-decode path */
  K3MOE_K_GEMM_GU = 5,  /* gate/up + SwiGLU, tcgen05 grouped GEMM */
  K3MOE_K_GEMM_DN = 6,  /* down projection, tcgen05 grouped GEMM */
  K3MOE_K_COMBINE = 7,  /* slot-ordered combine (both paths) */
  K3MOE_K_GATHER = 8,   /* activation preparation: h -> fp16 (both paths), x gather (GEMM path),
                           x fragments after the tensor-core router */
  K3MOE_K_COUNT = 9
};
typedef struct {
  double ms_total;
  long long launches;
} k3moe_kernel_time;
int k3moe_profile(k3moe_layer* layer, int enable);
int k3moe_profile_read(k3moe_layer* layer, k3moe_kernel_time* out);

/* Copy expert e's packed bytes (k3moe_packed_expert_bytes) to host memory `dst`;
 * synchronous.  For layout checks. */
int k3moe_read_packed(k3moe_layer* layer, int e, void* dst);

/* Diagnostics: device address and size of an internal buffer of the last call (read only;
 * valid until the layer's next call or free).  which: 0 = SwiGLU output h, fp32 [T_max*k][f];
 * 1 = per-pick expert outputs times the combine weight, fp32 [T_max*k][d]; 2 = the routed
 * expert ids, int32 [T_max][k]. */
int k3moe_debug_buffer(k3moe_layer* layer, int which, void** dev_ptr, size_t* bytes);

void k3moe_layer_free(k3moe_layer* layer);

/* Expert cache ("four reductions", expert LRU paragraph).  budget_bytes of device memory
 * are split into floor(budget/slot_bytes) slots, each holding one packed expert;
 * slot_bytes must equal k3moe_packed_expert_bytes of the layers that use the cache.
 * Least-recently-used experts are replaced; misses are copied from the layer's pinned pool
 * on a side stream.  Errors: INVALID_ARG (budget < one slot), OOM, CUDA. */
int k3moe_cache_create(size_t budget_bytes, size_t slot_bytes, k3moe_cache** out);
/* Keep the cache's LRU state on the device instead of the host (enable = 1; allowed only while no
 * layer uses the cache).  A layer call then looks its experts up with a one-thread kernel on its
 * own stream right after routing and copies the misses into their slots with the zero-copy kernel
 * (the SMs read the layer's mapped pinned pool): no host round trip between routing and the FFN,
 * so cache-mode calls queue like device-resident ones.  The policy and the statistics are those of
 * the host bookkeeping (hits made most recently used first, then each miss takes the least
 * recently used slot).  Because the device lookup cannot refuse a call, a layer attaches only when
 * min(E, T_max * k) <= slots (else K3MOE_ERR_BUDGET_TOO_SMALL from k3moe_pack_experts,
 * k3moe_layer_from_packed or k3moe_layer_set_cache).  Calls of layers sharing one cache must be
 * ordered (one stream).  K3MOE_OPT_MISS_PATH does not apply.  Errors: INVALID_ARG (NULL, layers
 * attached), OOM, CUDA. */
int k3moe_cache_set_device_lru(k3moe_cache* cache, int enable);
/* Waits for the layer calls it counts (a device synchronisation when some calls skipped the
 * lookup: their expert counts are read back asynchronously). */
int k3moe_cache_stats(const k3moe_cache* cache, k3moe_cache_stats_t* out);
int k3moe_cache_reset_stats(k3moe_cache* cache);
/* Destroy after every layer that uses it has been freed or moved to another cache. */
void k3moe_cache_destroy(k3moe_cache* cache);
/* Prefetch ("four reductions", expert LRU paragraph: the engine's cache loads the experts a
 * batch needs ahead of the arithmetic).  Makes experts[0..n) of `layer` resident in its cache
 * before a later call asks for them, so that the copies overlap work already queued:
 *   experts  host int32 [n], ids in 0..E-1 (duplicates allowed); n >= 0
 *   fetched  host int (may be NULL): the number of experts this call copied
 * Listed experts already resident become most recently used.  Each other listed expert, in list
 * order, takes the least recently used slot and is copied from the layer's pinned pool on the
 * cache's copy stream; this call does not wait for the copies.  A slot that a layer call still in
 * flight may read is never taken, nor one holding an expert the list names: the prefetch stops
 * at the first such slot, and `fetched` tells how far it got.  A call is known to have finished
 * once a later call of a layer on this cache has looked up its experts (that lookup waits for the
 * stream) or after k3moe_sync.  The next
 * layer call that uses a prefetched expert waits on its stream for the prefetch copies; its
 * output is unchanged (only which copies run, and when, differs).  Relies on the layers that
 * share a cache making their calls on one stream.  Errors: INVALID_ARG (NULL layer, a layer
 * without a cache, n < 0, experts NULL with n > 0, an id out of range: nothing is done),
 * UNSUPPORTED (the cache keeps its LRU state on the device), CUDA (a copy could not be issued:
 * its slot is forgotten, the copies issued before it stay valid). */
int k3moe_cache_prefetch(k3moe_layer* layer, const int32_t* experts, int n, int* fetched);
/* Moves a layer packed in cache mode (its experts in a pinned host pool) to another cache
 * with the same slot_bytes, e.g. to run the same layers under a different memory budget.
 * Waits for the layer's last stream, then drops the layer's experts from its old cache (its
 * next call misses on every expert).  The output of later calls is unchanged: the budget
 * changes only which copies run.  Errors: INVALID_ARG (NULL, a layer packed without a cache,
 * or slot_bytes differ), CUDA. */
int k3moe_layer_set_cache(k3moe_layer* layer, k3moe_cache* cache);

/* Cache-policy study ("four reductions", expert LRU paragraph, and the hit rates the pages
 * measure with a cache simulator on a recorded routing trace).  Host only: no device memory,
 * callable without a GPU.  Replays a trace of layer calls through n_slots expert slots:
 *   keys        host int64 [call_start[n_calls]]: the experts each call needs resident at once,
 *               any int64 that names an expert (e.g. layer * E + expert), distinct within a call,
 *               in the order the call looks them up (the device cache: ascending expert id)
 *   call_start  host int64 [n_calls + 1], call_start[0] = 0, non-decreasing: call c is
 *               keys[call_start[c] .. call_start[c+1])
 *   policy      K3MOE_POLICY_LRU: the device cache's policy (hits touched first, then each miss
 *               replaces the least recently used slot not touched by the call);
 *               K3MOE_POLICY_MIN: Belady's offline optimum (a miss in a full cache evicts the
 *               resident expert the call does not need whose next use is farthest ahead);
 *               K3MOE_POLICY_RANDOM: a miss in a full cache evicts a uniformly drawn resident
 *               expert the call does not need (splitmix64 stream seeded by `seed`)
 * Empty slots fill first (a miss, not an eviction).  out: hits + misses = call_start[n_calls].
 * Errors: INVALID_ARG (NULL pointers, n_slots < 1, bad call_start, a key repeated within a
 * call, unknown policy), BUDGET_TOO_SMALL (a call needs more than n_slots experts). */
#define K3MOE_POLICY_LRU 0
#define K3MOE_POLICY_MIN 1
#define K3MOE_POLICY_RANDOM 2
typedef struct {
  long long hits;
  long long misses;
  long long evictions;
} k3moe_cache_sim_stats;
int k3moe_cache_simulate(const int64_t* keys, const int64_t* call_start, int n_calls, int n_slots, int policy,
                         unsigned long long seed, k3moe_cache_sim_stats* out);

/* Glue between stacked layers (the layer's y excludes any residual).  For T tokens of
 * width d:  x_next = bf16_rne(x + y), the sum in fp32;  x_norm = bf16_rne(x_next /
 * sqrt(mean_j(x_next_j^2) + eps)), a weightless RMSNorm, the input a pre-norm block feeds
 * its next MoE layer.  The pages print no formula for it: the kimi-k3-in-c deep dive ("what
 * you learn", exercise paragraph) names the engine's RMSNorm kernel and its epsilon.
 *   y       device fp32 [T][d]                     (read)
 *   x       device bf16 bits [T][d]                (read; may alias x_next or x_norm)
 *   x_next  device bf16 bits [T][d]                (written)
 *   x_norm  device bf16 bits [T][d]                (written; must not alias x_next or y)
 * Asynchronous on `stream`.  Errors: INVALID_ARG (NULL, misaligned, T < 1, d < 1 or d > 65536,
 * eps < 0 or not finite, x_norm aliasing x_next), CUDA.  Non-finite sums propagate. */
int k3moe_residual_rmsnorm(const float* y, const void* x, int T, int d, float eps, void* x_next, void* x_norm,
                           void* stream);

const char* k3moe_last_error(void);

#ifdef __cplusplus
}
#endif
#endif
