// capi.cu -- the C ABI (include/k3moe.h): argument checks, ownership, workspace, dispatch,
// and the expert cache's host-side LRU bookkeeping.
#include <algorithm>
#include <cstdarg>
#include <cstddef>
#include <cstdio>
#include <cstring>
#include <iterator>
#include <list>
#include <unordered_map>
#include <utility>
#include <cmath>
#include <vector>

#include "k3moe_internal.cuh"

using namespace k3;

namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

#define CUDA_TRY(call)                                                                   \
  do {                                                                                   \
    cudaError_t e_ = (call);                                                             \
    if (e_ != cudaSuccess) return fail(K3MOE_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
  } while (0)

int check_dims(const k3moe_dims* d) {
  if (!d) return fail(K3MOE_ERR_INVALID_ARG, "dims is NULL");
  if (d->d <= 0 || d->d % 128 != 0 || d->d > 16384)
    return fail(K3MOE_ERR_INVALID_ARG, "d=%d must be a positive multiple of 128, <= 16384", d->d);
  if (d->f <= 0 || d->f % 128 != 0 || d->f > 16384)
    return fail(K3MOE_ERR_INVALID_ARG, "f=%d must be a positive multiple of 128, <= 16384", d->f);
  if (d->E < 1 || d->E > 4096) return fail(K3MOE_ERR_INVALID_ARG, "E=%d must be in 1..4096", d->E);
  if (d->k < 1 || d->k > d->E || d->k > 32)
    return fail(K3MOE_ERR_INVALID_ARG, "k=%d must be in 1..min(E, 32)", d->k);
  if (d->T_max < 1 || d->T_max > 65536) return fail(K3MOE_ERR_INVALID_ARG, "T_max=%d must be in 1..65536", d->T_max);
  return K3MOE_OK;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Copy raw bytes into the device (from host or device memory).
cudaError_t to_device(void* dst, const void* src, size_t n, int src_on_device, cudaStream_t s) {
  return cudaMemcpyAsync(dst, src, n, src_on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice, s);
}

struct TimedLaunch {
  int kid;
  cudaEvent_t a, b;
};

}  // namespace

void k3::set_last_error(const char* msg) { g_err = msg; }

struct k3moe_cache {
  size_t slot_bytes = 0;
  int n_slots = 0;
  uint8_t* slots = nullptr;
  cudaStream_t copy_stream = nullptr;
  std::list<int> lru;  // front = most recently used slot
  std::vector<std::list<int>::iterator> lru_pos;
  std::vector<long long> slot_key;  // (layer uid << 32) | expert, or -1 when empty
  std::unordered_map<long long, int> where;
  k3moe_cache_stats_t st{};
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> pending;  // copy timings not yet read
  std::vector<cudaEvent_t> free_events;
  int users = 0;
  int next_uid = 1;
  long long experts_attached = 0;         // experts of all layers using the cache
  std::unordered_map<int, int> resident;  // layer uid -> how many of its experts sit in slots
  // Calls that found every expert of their layer resident with nothing left to evict skip the
  // host lookup; their active-expert counts are read back asynchronously into this pinned ring
  // and added to the hit count by k3moe_cache_stats.
  static constexpr int kRing = 4096;
  int32_t* ring = nullptr;
  int ring_n = 0;
  // device-side LRU (k3moe_cache_set_device_lru): the state the lookup kernel keeps
  bool device_lru = false;
  LruState* d_state = nullptr;
  int32_t* d_prev = nullptr;
  int32_t* d_next = nullptr;
  int32_t** d_owner = nullptr;
  // Ordering of prefetches (k3moe_cache_prefetch) against the calls still in flight.  Calls get
  // increasing serials; a slot remembers the serial of the last call (or prefetch) that touched it.
  // The host LRU list, read from its back, holds the empty slots and then the filled ones in
  // nondecreasing serial, so the first slot a prefetch may not take ends its evictions.
  std::vector<long long> slot_call;
  long long calls_issued = 0;          // serial of the next call or prefetch
  long long done_before = 0;           // every call with a smaller serial has finished on the device
  bool fast_since_sync = false;        // a call skipped the lookup (touching no serial) since then
  cudaEvent_t prefetch_done = nullptr; // recorded on the copy stream after the last prefetch's copies
  bool prefetch_pending = false;
};

// Repeated layer calls captured as one CUDA graph (k3moe_graph_create).
struct k3moe_graph {
  k3moe_layer* layer = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
};

struct k3moe_layer {
  k3moe_dims dims{};
  size_t exp_bytes = 0;
  uint8_t* packed = nullptr;    // device, E * exp_bytes (device mode)
  uint8_t* pool = nullptr;      // pinned host, E * exp_bytes (cache mode); mapped
  uint8_t* pool_dev = nullptr;  // the pool's device address (zero-copy miss path)
  MissCopy* miss_host = nullptr;  // pinned [E]: a call's misses (zero-copy miss path)
  MissCopy* miss_dev = nullptr;   // device [E]
  int miss_path = K3MOE_MISS_COPY_ENGINE;
  int32_t* d_slot_of = nullptr;   // device [E]: expert -> slot (device-side LRU)
  int32_t* d_nmiss = nullptr;     // device [1]: the last call's misses (device-side LRU)
  float* Wr = nullptr;          // device [E][d]
  uint16_t* Wsplit = nullptr;   // device [E][2d] bf16: W_r rounded (hi) then the rounding remainder (lo)
  float* bias = nullptr;        // device [E] or nullptr
  const uint8_t** eptr_dev = nullptr;  // device [E]
  const uint8_t** eptr_host = nullptr; // pinned host [E] (cache mode staging)
  int32_t* act_host = nullptr;         // pinned host [E+1] (cache mode)
  void* ws_block = nullptr;
  Workspace ws;
  k3moe_cache* cache = nullptr;
  int uid = 0;
  int path = K3MOE_PATH_AUTO;
  long long router_tc_min_t = 64;  // from this many tokens the logits run on the tensor cores
  long long gemm_min_t = 512;  // AUTO: from this many tokens the tensor-core GEMM path
  bool profiling = false;
  std::vector<TimedLaunch> timed;
  std::vector<cudaEvent_t> spare_events;
  double prof_ms[K3MOE_K_COUNT] = {};
  long long prof_n[K3MOE_K_COUNT] = {};
  cudaStream_t last_stream = nullptr;
  cudaEvent_t copies_done = nullptr;
  uint16_t* x_stage = nullptr;  // forward_host staging
  float* y_stage = nullptr;
  uint32_t* flags_host = nullptr;  // pinned: device error flags read back by forward_host
  int num_sms = 148;
  unsigned long long wait_ns = 2000000000ull;  // bound on device-side waits
  int test_stall = 0;                           // next forward stalls its FFN consumers (timeout test)
  int test_fail_copy = 0;                       // n > 0: the n-th expert copy from now fails (test)
  int ring_depth = 0;                           // 0: automatic
  bool zero_scales = false;                     // some E8M0 scale byte is 0 (2^-127, a subnormal)
  int s_min = 255, s_max = 0;                   // range of the layer's scale bytes
  int activation = K3MOE_ACT_SWIGLU;            // gate activation of every expert
};

namespace {

cudaEvent_t take_event(k3moe_layer* L) {
  if (!L->spare_events.empty()) {
    cudaEvent_t e = L->spare_events.back();
    L->spare_events.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Launch helper: optional event pair around the launch, on the launch stream.
template <typename F>
int timed_launch(k3moe_layer* L, int kid, cudaStream_t s, F&& launch) {
  TimedLaunch tl{kid, nullptr, nullptr};
  if (L->profiling) {
    tl.a = take_event(L);
    tl.b = take_event(L);
    cudaEventRecord(tl.a, s);
  }
  cudaError_t e = launch();
  if (e != cudaSuccess) return fail(K3MOE_ERR_CUDA, "kernel %d launch: %s", kid, cudaGetErrorString(e));
  if (L->profiling) {
    cudaEventRecord(tl.b, s);
    L->timed.push_back(tl);
  }
  return K3MOE_OK;
}

int alloc_workspace(k3moe_layer* L) {
  const k3moe_dims& D = L->dims;
  const size_t T = D.T_max, P = (size_t)D.T_max * D.k;
  struct Item {
    void** dst;
    size_t bytes;
  };
  Workspace& w = L->ws;
  std::vector<Item> items = {
      {(void**)&w.logits, T * D.E * 4},  {(void**)&w.xfrag, T * D.d * 2},       {(void**)&w.xscale, T * 4},
      {(void**)&w.idx, P * 4},           {(void**)&w.w, P * 4},                 {(void**)&w.counts, (size_t)D.E * 4},
      {(void**)&w.offsets, (size_t)(D.E + 1) * 4}, {(void**)&w.perm, P * 4},    {(void**)&w.act, (size_t)D.E * 4},
      {(void**)&w.nact, 4},              {(void**)&w.units, (P / kUnitTokens + D.E + 1) * sizeof(UnitDesc)},
      {(void**)&w.nunits, 4},            {(void**)&w.hbuf, P * D.f * 4},
      {(void**)&w.hfrag, P * D.f * 2},   {(void**)&w.hscale, P * 4},
      {(void**)&w.obuf, P * D.d * 4},    {(void**)&w.sync, 64},                 {(void**)&w.bad, 16},
      {(void**)&w.hmax, P * 4},          {(void**)&w.mtiles, (P / 128 + D.E + 1) * sizeof(int4)},
      {(void**)&w.nmtiles, 4},           {(void**)&w.chist, (P / 2048 + 1) * D.E * 4},
  };
  size_t total = 0;
  for (auto& it : items) total += align256(it.bytes);
  if (cudaMalloc(&L->ws_block, total) != cudaSuccess) {
    cudaGetLastError();
    return fail(K3MOE_ERR_OOM, "workspace: cudaMalloc(%zu) failed", total);
  }
  size_t off = 0;
  for (auto& it : items) {
    *it.dst = (char*)L->ws_block + off;
    off += align256(it.bytes);
  }
  CUDA_TRY(cudaMemset(L->ws_block, 0, total));
  return K3MOE_OK;
}

// Adds the active-expert counts of the calls that skipped the lookup to the hit count.
cudaError_t fold_ring(k3moe_cache* C) {
  if (C->ring_n == 0) return cudaSuccess;
  const cudaError_t e = cudaDeviceSynchronize();  // the ring's copies ran on the layers' streams
  if (e != cudaSuccess) return e;
  for (int i = 0; i < C->ring_n; ++i) C->st.hits += (uint64_t)C->ring[i];
  C->ring_n = 0;
  return cudaSuccess;
}

// A timing event for the cache's copies: one from the pool, else a new one.
cudaEvent_t cache_event(k3moe_cache* C) {
  cudaEvent_t e = nullptr;
  if (!C->free_events.empty()) {
    e = C->free_events.back();
    C->free_events.pop_back();
  } else {
    cudaEventCreate(&e);
  }
  return e;
}

// The slot holds no valid expert (any more): it becomes empty and least recently used, so that
// no later call takes it for a hit and the next miss takes it first.
void forget_slot(k3moe_cache* C, int slot) {
  const long long key = C->slot_key[slot];
  if (key >= 0) {
    C->where.erase(key);
    C->resident[(int)(key >> 32)] -= 1;
  }
  C->slot_key[slot] = -1;
  C->lru.erase(C->lru_pos[slot]);
  C->lru.push_back(slot);
  C->lru_pos[slot] = std::prev(C->lru.end());
}

int attach_cache(k3moe_layer* L, k3moe_cache* C) {
  if (C->device_lru) {
    // the lookup kernel cannot refuse a call: every call must fit in the slots
    const long long need = std::min<long long>(L->dims.E, (long long)L->dims.T_max * L->dims.k);
    if (need > C->n_slots)
      return fail(K3MOE_ERR_BUDGET_TOO_SMALL, "a call may need %lld experts resident, the cache has %d slots", need,
                  C->n_slots);
    if (!L->d_slot_of && (cudaMalloc((void**)&L->d_slot_of, (size_t)L->dims.E * 4) != cudaSuccess ||
                          cudaMalloc((void**)&L->d_nmiss, 4) != cudaSuccess)) {
      cudaGetLastError();
      return fail(K3MOE_ERR_OOM, "device-side cache tables could not be allocated");
    }
    CUDA_TRY(cudaMemset(L->d_slot_of, 0xFF, (size_t)L->dims.E * 4));  // -1: not resident
  }
  L->cache = C;
  L->uid = C->next_uid++;
  C->users += 1;
  C->experts_attached += L->dims.E;
  C->resident[L->uid] = 0;
  return K3MOE_OK;
}

// Drops the layer's experts from its cache: their slots become free (least recently used).
void detach_cache(k3moe_layer* L) {
  k3moe_cache* C = L->cache;
  if (!C) return;
  if (C->device_lru && L->d_slot_of) {
    launch_lru_detach(C->d_state, C->d_prev, C->d_next, C->d_owner, C->n_slots, L->d_slot_of, L->dims.E, nullptr);
    cudaDeviceSynchronize();
  }
  fold_ring(C);
  C->experts_attached -= L->dims.E;
  for (int s = 0; s < C->n_slots; ++s)
    if (C->slot_key[s] >= 0 && (int)(C->slot_key[s] >> 32) == L->uid) forget_slot(C, s);
  C->resident.erase(L->uid);
  C->users -= 1;
  L->cache = nullptr;
}

void free_layer(k3moe_layer* L) {
  if (!L) return;
  if (L->last_stream) cudaStreamSynchronize(L->last_stream);
  cudaFree(L->packed);
  cudaFreeHost(L->pool);
  cudaFreeHost(L->miss_host);
  cudaFree(L->miss_dev);
  cudaFree(L->Wr);
  cudaFree(L->Wsplit);
  cudaFree(L->bias);
  cudaFree((void*)L->eptr_dev);
  cudaFreeHost((void*)L->eptr_host);
  cudaFreeHost(L->act_host);
  cudaFree(L->ws_block);
  cudaFree(L->x_stage);
  cudaFree(L->y_stage);
  cudaFreeHost(L->flags_host);
  for (auto& t : L->timed) {
    cudaEventDestroy(t.a);
    cudaEventDestroy(t.b);
  }
  for (auto e : L->spare_events) cudaEventDestroy(e);
  if (L->copies_done) cudaEventDestroy(L->copies_done);
  detach_cache(L);
  cudaFree(L->d_slot_of);
  cudaFree(L->d_nmiss);
  delete L;
}

// After a kernel gave up part-way, clear the error flags and the per-call counters that a
// completed call leaves at zero.
cudaError_t reset_after_timeout(k3moe_layer* L) {
  const k3moe_dims& D = L->dims;
  cudaError_t e = cudaMemset(L->ws.sync, 0, 64);
  if (e == cudaSuccess) e = cudaMemset(L->ws.hmax, 0, (size_t)D.T_max * D.k * 4);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  return e;
}

bool use_gemm(const k3moe_layer* L, int T) {
  if (L->path == K3MOE_PATH_GEMM) return true;
  if (L->path == K3MOE_PATH_DECODE) return false;
  return (long long)T >= L->gemm_min_t && gemm_scales_ok(L->s_min, L->s_max);
}

// Router + selection + bucketing into the workspace.  need_frag: the register-decode FFN
// follows, which needs the fp16 fragments of x.  From router_tc_min_t tokens the logits run on
// the tensor cores (and a small kernel writes the fragments when they are needed); below, the
// CUDA-core router kernel computes the logits and writes the fragments itself.
int run_routing(k3moe_layer* L, const void* x, int T, cudaStream_t s, bool need_frag) {
  const k3moe_dims& D = L->dims;
  RouterArgs ra{reinterpret_cast<const uint16_t*>(x), L->Wr, L->bias, T, D.d, D.E, D.k, L->ws, 0, need_frag ? 0 : 1};
  // the last router block selects serially token by token: worth it only for a few tokens
  ra.fuse_select = (T <= 4 && T * D.k <= 1024) ? 1 : 0;
  const bool tc = !ra.fuse_select && (long long)T >= L->router_tc_min_t && (reinterpret_cast<uintptr_t>(x) & 15u) == 0;
  int rc = tc ? timed_launch(L, KID_ROUTER, s,
                             [&] {
                               return launch_router_tc(reinterpret_cast<const uint16_t*>(x), T, D.d, D.E, L->Wsplit,
                                                       L->ws.logits, L->ws.sync + 1, L->wait_ns, L->num_sms, s);
                             })
              : timed_launch(L, KID_ROUTER, s, [&] { return launch_router(ra, s); });
  if (rc) return rc;
  if (tc && need_frag) {
    rc = timed_launch(L, KID_GATHER, s, [&] { return launch_convert(ra, L->num_sms, s); });
    if (rc) return rc;
  }
  if (!ra.fuse_select) {
    rc = timed_launch(L, KID_TOPK, s,
                      [&] { return launch_topk(L->ws.logits, L->bias, T, D.E, D.k, L->ws.idx, L->ws.w, s); });
    if (rc) return rc;
    rc = timed_launch(L, KID_BUCKET, s, [&] {
      return launch_bucket(L->ws.idx, T, D.k, D.E, L->ws.counts, L->ws.offsets, L->ws.perm, L->ws.act, L->ws.nact,
                           L->ws.units, L->ws.nunits, L->ws.w, L->ws.xscale, L->ws.chist, s, need_frag);
    });
    if (rc) return rc;
  }
  return K3MOE_OK;
}

// Cache mode: make every active expert resident; fill eptr_dev for them.
int make_resident(k3moe_layer* L, cudaStream_t s) {
  k3moe_cache* C = L->cache;
  const int E = L->dims.E;
  if (C->device_lru) {
    // lookup and copies on the device, on `s`: no host round trip
    LruArgs la{C->d_state, C->d_prev, C->d_next, C->d_owner, C->n_slots, C->slots, C->slot_bytes, L->ws.act,
               L->ws.nact, L->d_slot_of, (const uint8_t**)L->eptr_dev, L->pool_dev, L->miss_dev, L->d_nmiss,
               L->ws.sync + 1};
    cudaEvent_t a = cache_event(C), b = cache_event(C);
    CUDA_TRY(launch_lru_lookup(la, s));
    CUDA_TRY(cudaEventRecord(a, s));
    CUDA_TRY(launch_miss_copy_dev(L->miss_dev, L->d_nmiss, std::min(E, L->dims.T_max * L->dims.k), L->exp_bytes,
                                  L->num_sms, s));
    CUDA_TRY(cudaEventRecord(b, s));
    C->pending.emplace_back(a, b);
    return K3MOE_OK;
  }
  if ((long long)C->n_slots >= C->experts_attached && C->resident[L->uid] == E) {
    // every expert of the layer has a slot and nothing can be evicted: the pointer table on
    // the device is complete, so no lookup (and no host round trip) is needed
    if (C->ring_n == k3moe_cache::kRing) CUDA_TRY(fold_ring(C));
    CUDA_TRY(cudaMemcpyAsync(C->ring + C->ring_n, L->ws.nact, 4, cudaMemcpyDeviceToHost, s));
    C->ring_n += 1;
    C->st.calls += 1;
    C->calls_issued += 1;
    C->fast_since_sync = true;
    if (C->prefetch_pending) CUDA_TRY(cudaStreamWaitEvent(s, C->prefetch_done, 0));  // a prefetched slot
    return K3MOE_OK;
  }
  CUDA_TRY(cudaMemcpyAsync(L->act_host, L->ws.nact, 4, cudaMemcpyDeviceToHost, s));
  CUDA_TRY(cudaMemcpyAsync(L->act_host + 1, L->ws.act, (size_t)E * 4, cudaMemcpyDeviceToHost, s));
  CUDA_TRY(cudaStreamSynchronize(s));
  // every earlier call (one stream) has finished: their slots are free for a prefetch to take
  const long long serial = C->calls_issued++;
  C->done_before = serial;
  C->fast_since_sync = false;
  if (C->prefetch_pending) {
    // this call's hits, and the slots its misses take, may still be receiving prefetch copies
    if (cudaEventQuery(C->prefetch_done) == cudaSuccess)
      C->prefetch_pending = false;
    else
      CUDA_TRY(cudaStreamWaitEvent(s, C->prefetch_done, 0));
  }
  const int nact = L->act_host[0];
  if (nact < 0 || nact > E) return fail(K3MOE_ERR_CUDA, "corrupt active-expert count %d", nact);
  if (nact > C->n_slots)
    return fail(K3MOE_ERR_BUDGET_TOO_SMALL, "call needs %d experts resident, cache has %d slots", nact, C->n_slots);
  const int32_t* act = L->act_host + 1;
  // pass 1: hits are touched first so that no expert of this call is evicted
  std::vector<int> miss;
  for (int i = 0; i < nact; ++i) {
    const long long key = ((long long)L->uid << 32) | act[i];
    auto it = C->where.find(key);
    if (it != C->where.end()) {
      const int slot = it->second;
      C->lru.erase(C->lru_pos[slot]);
      C->lru.push_front(slot);
      C->lru_pos[slot] = C->lru.begin();
      C->slot_call[slot] = serial;
      L->eptr_host[act[i]] = C->slots + (size_t)slot * C->slot_bytes;
      C->st.hits += 1;
    } else {
      miss.push_back(act[i]);
    }
  }
  if (!miss.empty()) {
    cudaEvent_t a = cache_event(C), b = cache_event(C);
    const bool zc = L->miss_path == K3MOE_MISS_ZERO_COPY;
    if (zc) {
      // the copy kernel runs on `s` itself, after every earlier use of the slots on `s`
      CUDA_TRY(cudaEventRecord(a, s));
    } else {
      // the copy stream must not overwrite a slot that earlier queued work on `s` may still read
      CUDA_TRY(cudaEventRecord(L->copies_done, s));
      CUDA_TRY(cudaStreamWaitEvent(C->copy_stream, L->copies_done, 0));
      CUDA_TRY(cudaEventRecord(a, C->copy_stream));
    }
    int nm = 0;           // zero-copy: misses listed for the copy kernel
    int failed_e = -1;    // the miss whose copy failed, if any
    cudaError_t failed_ce = cudaSuccess;
    for (int e : miss) {
      const int slot = C->lru.back();  // least recently used; never one touched in pass 1
      C->lru.pop_back();
      if (C->slot_key[slot] >= 0) {
        C->where.erase(C->slot_key[slot]);
        C->st.evictions += 1;
        C->resident[(int)(C->slot_key[slot] >> 32)] -= 1;
      }
      C->resident[L->uid] += 1;
      const long long key = ((long long)L->uid << 32) | e;
      C->slot_key[slot] = key;
      C->where[key] = slot;
      C->lru.push_front(slot);
      C->lru_pos[slot] = C->lru.begin();
      C->slot_call[slot] = serial;
      uint8_t* dst = C->slots + (size_t)slot * C->slot_bytes;
      const bool fake = L->test_fail_copy > 0 && --L->test_fail_copy == 0;  // failure-path test
      cudaError_t ce = cudaSuccess;
      if (fake)
        ce = cudaErrorInvalidValue;
      else if (zc)
        L->miss_host[nm++] = MissCopy{L->pool_dev + (size_t)e * L->exp_bytes, dst};
      else
        ce = cudaMemcpyAsync(dst, L->pool + (size_t)e * L->exp_bytes, L->exp_bytes, cudaMemcpyHostToDevice,
                             C->copy_stream);
      if (ce != cudaSuccess) {
        if (!fake) cudaGetLastError();
        // the slot holds no valid expert: forget it; the copies issued before it still complete,
        // and later work on `s` is ordered after them
        forget_slot(C, slot);
        failed_e = e;
        failed_ce = ce;
        break;
      }
      L->eptr_host[e] = dst;
      C->st.misses += 1;
      C->st.h2d_bytes += L->exp_bytes;
    }
    if (zc) {
      cudaError_t ke = cudaSuccess;
      if (nm > 0) ke = cudaMemcpyAsync(L->miss_dev, L->miss_host, (size_t)nm * sizeof(MissCopy), cudaMemcpyHostToDevice, s);
      if (ke == cudaSuccess) ke = launch_miss_copy(L->miss_dev, nm, L->exp_bytes, L->num_sms, s);
      cudaEventRecord(b, s);
      C->pending.emplace_back(a, b);
      if (ke != cudaSuccess) {
        cudaGetLastError();
        // none of this call's slots was filled: forget them all
        for (int i = 0; i < nm; ++i) forget_slot(C, (int)((L->miss_host[i].dst - C->slots) / C->slot_bytes));
        return fail(K3MOE_ERR_CUDA, "zero-copy miss kernel: %s", cudaGetErrorString(ke));
      }
    } else {
      cudaEventRecord(b, C->copy_stream);
      C->pending.emplace_back(a, b);
      cudaStreamWaitEvent(s, b, 0);
    }
    if (failed_e >= 0) {
      cudaMemcpyAsync((void*)L->eptr_dev, L->eptr_host, (size_t)E * sizeof(void*), cudaMemcpyHostToDevice, s);
      return fail(K3MOE_ERR_CUDA, "copying expert %d to its cache slot failed: %s", failed_e,
                  cudaGetErrorString(failed_ce));
    }
  }
  C->st.calls += 1;
  CUDA_TRY(cudaMemcpyAsync((void*)L->eptr_dev, L->eptr_host, (size_t)E * sizeof(void*), cudaMemcpyHostToDevice, s));
  return K3MOE_OK;
}

// Large T: the tcgen05 grouped GEMM path (gemm_tc.cu), then the slot-ordered combine.
int forward_gemm(k3moe_layer* L, const void* x, int T, float* y, cudaStream_t s) {
  const k3moe_dims& D = L->dims;
  int rc = run_routing(L, x, T, s, false);
  if (rc) return rc;
  if (L->cache) {
    rc = make_resident(L, s);
    if (rc) return rc;
  }
  Workspace& w = L->ws;
  const int P = T * D.k;
  GemmFfn q{};
  q.expert_ptr = L->eptr_dev;
  q.d = D.d;
  q.f = D.f;
  q.k = D.k;
  q.T = T;
  q.s_ref = L->s_max - 13;
  q.wscale = std::ldexp(1.0f, q.s_ref - 127);
  q.mtiles = w.mtiles;
  q.nmtiles = w.nmtiles;
  q.perm = w.perm;
  q.w = w.w;
  q.xs = w.xscale;
  q.xg = reinterpret_cast<__half*>(w.obuf);
  q.hbuf = w.hbuf;
  q.hmax = w.hmax;
  q.h16 = w.hfrag;
  q.hs = w.hscale;
  q.obuf = w.obuf;
  q.err = w.sync + 1;
  q.wait_ns = L->wait_ns;
  q.num_sms = L->num_sms;
  q.act = L->activation;
  rc = timed_launch(L, KID_GATHER, s, [&] {
    cudaError_t e = launch_gemm_prep(q, reinterpret_cast<const uint16_t*>(x), w.counts, w.offsets, D.E, s);
    return e == cudaSuccess ? cudaMemsetAsync(w.hmax, 0, (size_t)P * 4, s) : e;
  });
  if (rc) return rc;
  rc = timed_launch(L, KID_GEMM_GU, s, [&] { return launch_gemm_gu(q, s); });
  if (rc) return rc;
  rc = timed_launch(L, KID_GATHER, s, [&] { return launch_gemm_h16(q, P, s); });
  if (rc) return rc;
  rc = timed_launch(L, KID_GEMM_DN, s, [&] { return launch_gemm_dn(q, s); });
  if (rc) return rc;
  FfnArgs fa{L->eptr_dev, D.d, D.f, D.E, D.k, T, L->ws, y, L->num_sms, L->wait_ns, 0, 0, 0, nullptr, 0, L->activation};
  return timed_launch(L, KID_COMBINE, s, [&] { return launch_combine(fa, s); });
}

int forward_impl(k3moe_layer* L, const void* x, int T, float* y, cudaStream_t s) {
  const k3moe_dims& D = L->dims;
  L->last_stream = s;
  if (use_gemm(L, T)) {
    if (!gemm_scales_ok(L->s_min, L->s_max))
      return fail(K3MOE_ERR_UNSUPPORTED,
                  "scale bytes span %d..%d: wider than the 36 steps the fp16 tensor-core path holds exactly",
                  L->s_min, L->s_max);
    return forward_gemm(L, x, T, y, s);
  }
  int rc = run_routing(L, x, T, s, true);
  if (rc) return rc;
  if (L->cache) {
    rc = make_resident(L, s);
    if (rc) return rc;
  }
  FfnArgs fa{L->eptr_dev, D.d, D.f, D.E, D.k, T, L->ws, y, L->num_sms, L->wait_ns, L->test_stall, L->ring_depth,
             L->zero_scales ? 1 : 0, L->cache ? nullptr : L->packed, L->exp_bytes, L->activation};
  L->test_stall = 0;
  rc = timed_launch(L, KID_GATEUP, s, [&] { return launch_gateup(fa, s); });
  if (rc) return rc;
  rc = timed_launch(L, KID_GATHER, s, [&] { return launch_hconv(fa, s); });
  if (rc) return rc;
  rc = timed_launch(L, KID_DOWN, s, [&] { return launch_down(fa, s); });
  if (rc) return rc;
  return timed_launch(L, KID_COMBINE, s, [&] { return launch_combine(fa, s); });
}

}  // namespace

extern "C" {

size_t k3moe_packed_expert_bytes(const k3moe_dims* dims) {
  if (check_dims(dims) != K3MOE_OK) return 0;
  return packed_expert_bytes(dims->d, dims->f);
}

const char* k3moe_last_error(void) { return g_err.c_str(); }

int k3moe_cache_create(size_t budget_bytes, size_t slot_bytes, k3moe_cache** out) {
  if (!out) return fail(K3MOE_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (slot_bytes == 0 || slot_bytes % 256 != 0)
    return fail(K3MOE_ERR_INVALID_ARG, "slot_bytes=%zu must be a positive multiple of 256", slot_bytes);
  if (budget_bytes < slot_bytes)
    return fail(K3MOE_ERR_INVALID_ARG, "budget %zu bytes is smaller than one slot (%zu)", budget_bytes, slot_bytes);
  const size_t n = budget_bytes / slot_bytes;
  if (n > (1u << 30)) return fail(K3MOE_ERR_INVALID_ARG, "too many slots");
  k3moe_cache* C = new k3moe_cache();
  C->slot_bytes = slot_bytes;
  C->n_slots = (int)n;
  if (cudaMalloc(&C->slots, n * slot_bytes) != cudaSuccess) {
    cudaGetLastError();
    delete C;
    return fail(K3MOE_ERR_OOM, "cache: cudaMalloc(%zu) failed", n * slot_bytes);
  }
  if (cudaStreamCreateWithFlags(&C->copy_stream, cudaStreamNonBlocking) != cudaSuccess) {
    cudaFree(C->slots);
    delete C;
    return fail(K3MOE_ERR_CUDA, "cache: stream creation failed");
  }
  if (cudaHostAlloc((void**)&C->ring, k3moe_cache::kRing * sizeof(int32_t), cudaHostAllocDefault) != cudaSuccess) {
    cudaGetLastError();
    cudaStreamDestroy(C->copy_stream);
    cudaFree(C->slots);
    delete C;
    return fail(K3MOE_ERR_OOM, "cache: pinned counter ring allocation failed");
  }
  C->lru_pos.resize(n);
  C->slot_key.assign(n, -1);
  C->slot_call.assign(n, -1);
  for (int i = 0; i < (int)n; ++i) {
    C->lru.push_back(i);
    C->lru_pos[i] = std::prev(C->lru.end());
  }
  *out = C;
  return K3MOE_OK;
}

int k3moe_cache_stats(const k3moe_cache* cc, k3moe_cache_stats_t* out) {
  if (!cc || !out) return fail(K3MOE_ERR_INVALID_ARG, "NULL argument");
  k3moe_cache* C = const_cast<k3moe_cache*>(cc);
  CUDA_TRY(fold_ring(C));
  if (C->device_lru) {
    LruState st;
    CUDA_TRY(cudaDeviceSynchronize());
    CUDA_TRY(cudaMemcpy(&st, C->d_state, sizeof(st), cudaMemcpyDeviceToHost));
    C->st.hits = st.hits;
    C->st.misses = st.misses;
    C->st.evictions = st.evictions;
    C->st.calls = st.calls;
    C->st.h2d_bytes = st.misses * C->slot_bytes;
  }
  for (auto& pr : C->pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(pr.second) == cudaSuccess && cudaEventElapsedTime(&ms, pr.first, pr.second) == cudaSuccess)
      C->st.h2d_ms += ms;
    C->free_events.push_back(pr.first);
    C->free_events.push_back(pr.second);
  }
  C->pending.clear();
  *out = C->st;
  return K3MOE_OK;
}

int k3moe_cache_reset_stats(k3moe_cache* C) {
  if (!C) return fail(K3MOE_ERR_INVALID_ARG, "cache is NULL");
  k3moe_cache_stats_t tmp;
  k3moe_cache_stats(C, &tmp);
  C->st = k3moe_cache_stats_t{};
  if (C->device_lru) {
    LruState st;
    CUDA_TRY(cudaMemcpy(&st, C->d_state, sizeof(st), cudaMemcpyDeviceToHost));
    st.hits = st.misses = st.evictions = st.calls = 0;
    CUDA_TRY(cudaMemcpy(C->d_state, &st, sizeof(st), cudaMemcpyHostToDevice));
  }
  return K3MOE_OK;
}

void k3moe_cache_destroy(k3moe_cache* C) {
  if (!C) return;
  if (C->copy_stream) {
    cudaStreamSynchronize(C->copy_stream);
    cudaStreamDestroy(C->copy_stream);
  }
  for (auto& pr : C->pending) {
    cudaEventDestroy(pr.first);
    cudaEventDestroy(pr.second);
  }
  for (auto e : C->free_events) cudaEventDestroy(e);
  if (C->prefetch_done) cudaEventDestroy(C->prefetch_done);
  cudaFree(C->slots);
  cudaFreeHost(C->ring);
  cudaFree(C->d_state);
  cudaFree(C->d_prev);
  cudaFree(C->d_next);
  cudaFree((void*)C->d_owner);
  delete C;
}

int k3moe_cache_set_device_lru(k3moe_cache* C, int enable) {
  if (!C) return fail(K3MOE_ERR_INVALID_ARG, "cache is NULL");
  if (enable != 0 && enable != 1) return fail(K3MOE_ERR_INVALID_ARG, "enable must be 0 or 1");
  if (C->users != 0) return fail(K3MOE_ERR_INVALID_ARG, "the cache already serves %d layers", C->users);
  if ((enable != 0) == C->device_lru) return K3MOE_OK;
  if (!enable) {
    cudaFree(C->d_state);
    cudaFree(C->d_prev);
    cudaFree(C->d_next);
    cudaFree((void*)C->d_owner);
    C->d_state = nullptr;
    C->d_prev = C->d_next = nullptr;
    C->d_owner = nullptr;
    C->device_lru = false;
    return K3MOE_OK;
  }
  const int n = C->n_slots;
  if (cudaMalloc((void**)&C->d_state, sizeof(LruState)) != cudaSuccess ||
      cudaMalloc((void**)&C->d_prev, (size_t)n * 4) != cudaSuccess ||
      cudaMalloc((void**)&C->d_next, (size_t)n * 4) != cudaSuccess ||
      cudaMalloc((void**)&C->d_owner, (size_t)n * sizeof(int32_t*)) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(C->d_state);
    cudaFree(C->d_prev);
    cudaFree(C->d_next);
    C->d_state = nullptr;
    C->d_prev = C->d_next = nullptr;
    return fail(K3MOE_ERR_OOM, "device-side cache state could not be allocated");
  }
  // the host bookkeeping's initial order: slot 0 most recently used ... slot n-1 least
  std::vector<int32_t> prev(n), next(n);
  for (int i = 0; i < n; ++i) {
    prev[i] = i - 1;
    next[i] = i + 1 < n ? i + 1 : -1;
  }
  LruState st{0, n - 1, 0, 0, 0, 0};
  CUDA_TRY(cudaMemcpy(C->d_prev, prev.data(), (size_t)n * 4, cudaMemcpyHostToDevice));
  CUDA_TRY(cudaMemcpy(C->d_next, next.data(), (size_t)n * 4, cudaMemcpyHostToDevice));
  CUDA_TRY(cudaMemset((void*)C->d_owner, 0, (size_t)n * sizeof(int32_t*)));
  CUDA_TRY(cudaMemcpy(C->d_state, &st, sizeof(st), cudaMemcpyHostToDevice));
  C->device_lru = true;
  return K3MOE_OK;
}

int k3moe_cache_prefetch(k3moe_layer* L, const int32_t* experts, int n, int* fetched) {
  if (fetched) *fetched = 0;
  if (!L) return fail(K3MOE_ERR_INVALID_ARG, "layer is NULL");
  k3moe_cache* C = L->cache;
  if (!C) return fail(K3MOE_ERR_INVALID_ARG, "the layer has no cache: its experts are device-resident");
  if (C->device_lru)
    return fail(K3MOE_ERR_UNSUPPORTED, "prefetch needs the host-side LRU bookkeeping (the cache keeps it on the device)");
  if (n < 0 || (n > 0 && !experts)) return fail(K3MOE_ERR_INVALID_ARG, "bad expert list (n=%d)", n);
  const int E = L->dims.E;
  for (int i = 0; i < n; ++i)
    if (experts[i] < 0 || experts[i] >= E)
      return fail(K3MOE_ERR_INVALID_ARG, "experts[%d]=%d is not in 0..%d", i, experts[i], E - 1);
  // a prefetch takes a serial like a call: the slots it touches are not taken by a later prefetch
  // before a call (or k3moe_sync) has waited for the work queued up to here
  const long long serial = C->calls_issued++;
  auto may_take = [&](int slot) {
    return C->slot_key[slot] < 0 || (!C->fast_since_sync && C->slot_call[slot] < C->done_before);
  };
  for (int i = 0; i < n; ++i) {
    auto it = C->where.find(((long long)L->uid << 32) | experts[i]);
    if (it == C->where.end()) continue;
    const int slot = it->second;
    C->lru.erase(C->lru_pos[slot]);
    C->lru.push_front(slot);
    C->lru_pos[slot] = C->lru.begin();
    C->slot_call[slot] = std::max(C->slot_call[slot], serial);
  }
  int got = 0;
  int failed_e = -1;
  cudaError_t failed_ce = cudaSuccess;
  cudaEvent_t a = nullptr;
  for (int i = 0; i < n; ++i) {
    const int e = experts[i];
    const long long key = ((long long)L->uid << 32) | e;
    if (C->where.count(key)) continue;  // resident, or listed twice
    const int slot = C->lru.back();
    if (!may_take(slot)) break;  // every slot nearer the front was touched later: in flight too
    if (!a) {
      // the copies need no wait on a compute stream: no call in flight reads the slots they fill
      a = cache_event(C);
      CUDA_TRY(cudaEventRecord(a, C->copy_stream));
    }
    C->lru.pop_back();
    if (C->slot_key[slot] >= 0) {
      C->where.erase(C->slot_key[slot]);
      C->st.evictions += 1;
      C->resident[(int)(C->slot_key[slot] >> 32)] -= 1;
    }
    C->resident[L->uid] += 1;
    C->slot_key[slot] = key;
    C->where[key] = slot;
    C->lru.push_front(slot);
    C->lru_pos[slot] = C->lru.begin();
    C->slot_call[slot] = serial;
    uint8_t* dst = C->slots + (size_t)slot * C->slot_bytes;
    const bool fake = L->test_fail_copy > 0 && --L->test_fail_copy == 0;  // failure-path test
    const cudaError_t ce = fake ? cudaErrorInvalidValue
                                : cudaMemcpyAsync(dst, L->pool + (size_t)e * L->exp_bytes, L->exp_bytes,
                                                  cudaMemcpyHostToDevice, C->copy_stream);
    if (ce != cudaSuccess) {
      if (!fake) cudaGetLastError();
      forget_slot(C, slot);
      failed_e = e;
      failed_ce = ce;
      break;
    }
    got += 1;
    C->st.prefetched += 1;
    C->st.h2d_bytes += L->exp_bytes;
  }
  if (a) {
    cudaEvent_t b = cache_event(C);
    CUDA_TRY(cudaEventRecord(b, C->copy_stream));
    C->pending.emplace_back(a, b);
    if (!C->prefetch_done) CUDA_TRY(cudaEventCreateWithFlags(&C->prefetch_done, cudaEventDisableTiming));
    CUDA_TRY(cudaEventRecord(C->prefetch_done, C->copy_stream));
    C->prefetch_pending = true;
  }
  if (fetched) *fetched = got;
  if (failed_e >= 0)
    return fail(K3MOE_ERR_CUDA, "prefetching expert %d into its cache slot failed: %s", failed_e,
                cudaGetErrorString(failed_ce));
  return K3MOE_OK;
}

}  // extern "C"

namespace {

// A layer with everything but its expert bytes: workspace, router (and its bf16 split), pointer
// table, and the storage the experts will fill (the device block, or in cache mode the mapped
// pinned pool and its host-side tables).  On failure nothing is left allocated.
int layer_begin(const k3moe_dims* dims, int src_on_device, const float* W_r, const float* bias, k3moe_cache* cache,
                cudaStream_t s, k3moe_layer** out) {
  *out = nullptr;
  int rc = check_dims(dims);
  if (rc) return rc;
  if (!W_r) return fail(K3MOE_ERR_INVALID_ARG, "NULL input pointer");
  if (src_on_device != 0 && src_on_device != 1) return fail(K3MOE_ERR_INVALID_ARG, "src_on_device must be 0 or 1");
  const k3moe_dims D = *dims;
  const size_t eb = packed_expert_bytes(D.d, D.f);
  if (cache && cache->slot_bytes != eb)
    return fail(K3MOE_ERR_INVALID_ARG, "cache slot_bytes %zu != packed expert bytes %zu", cache->slot_bytes, eb);
  k3moe_layer* L = new k3moe_layer();
  L->dims = D;
  L->exp_bytes = eb;
  L->cache = cache;
  {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
        n > 0)
      L->num_sms = n;
    cudaGetLastError();
  }
  auto bail = [&](int code) {
    L->cache = nullptr;  // not attached yet
    free_layer(L);
    return code;
  };
  if ((rc = alloc_workspace(L))) return bail(rc);
  if (cudaEventCreateWithFlags(&L->copies_done, cudaEventDisableTiming) != cudaSuccess)
    return bail(fail(K3MOE_ERR_CUDA, "event creation failed"));
  if (cudaMalloc(&L->Wr, (size_t)D.E * D.d * 4) != cudaSuccess ||
      (bias && cudaMalloc(&L->bias, (size_t)D.E * 4) != cudaSuccess) ||
      cudaMalloc((void**)&L->eptr_dev, (size_t)D.E * sizeof(void*)) != cudaSuccess) {
    cudaGetLastError();
    return bail(fail(K3MOE_ERR_OOM, "router/pointer table allocation failed"));
  }
  if (to_device(L->Wr, W_r, (size_t)D.E * D.d * 4, src_on_device, s) != cudaSuccess ||
      (bias && to_device(L->bias, bias, (size_t)D.E * 4, src_on_device, s) != cudaSuccess))
    return bail(fail(K3MOE_ERR_CUDA, "router copy failed: %s", cudaGetErrorString(cudaGetLastError())));
  if (cudaMalloc(&L->Wsplit, (size_t)D.E * D.d * 4) != cudaSuccess) {
    cudaGetLastError();
    return bail(fail(K3MOE_ERR_OOM, "router split weights allocation failed"));
  }
  if (launch_split_router(L->Wr, D.E, D.d, L->Wsplit, s) != cudaSuccess)
    return bail(fail(K3MOE_ERR_CUDA, "router split failed: %s", cudaGetErrorString(cudaGetLastError())));
  if (!cache) {
    if (cudaMalloc(&L->packed, (size_t)D.E * eb) != cudaSuccess) {
      cudaGetLastError();
      return bail(fail(K3MOE_ERR_OOM, "packed experts: cudaMalloc(%zu) failed", (size_t)D.E * eb));
    }
  } else {
    if (cudaHostAlloc(&L->pool, (size_t)D.E * eb, cudaHostAllocMapped) != cudaSuccess ||
        cudaHostGetDevicePointer((void**)&L->pool_dev, L->pool, 0) != cudaSuccess ||
        cudaHostAlloc((void**)&L->miss_host, (size_t)D.E * sizeof(MissCopy), cudaHostAllocDefault) != cudaSuccess ||
        cudaMalloc((void**)&L->miss_dev, (size_t)D.E * sizeof(MissCopy)) != cudaSuccess ||
        cudaHostAlloc((void**)&L->eptr_host, (size_t)D.E * sizeof(void*), cudaHostAllocDefault) != cudaSuccess ||
        cudaHostAlloc((void**)&L->act_host, (size_t)(D.E + 1) * 4, cudaHostAllocDefault) != cudaSuccess) {
      cudaGetLastError();
      return bail(fail(K3MOE_ERR_OOM, "pinned expert pool of %zu bytes could not be allocated", (size_t)D.E * eb));
    }
    memset((void*)L->eptr_host, 0, (size_t)D.E * sizeof(void*));
  }
  *out = L;
  return K3MOE_OK;
}

// The experts are in place: fill the device pointer table (device mode) or attach to the cache.
int layer_finish(k3moe_layer* L, cudaStream_t s) {
  const k3moe_dims& D = L->dims;
  if (!L->cache) {
    std::vector<const uint8_t*> ptrs(D.E);
    for (int e = 0; e < D.E; ++e) ptrs[e] = L->packed + (size_t)e * L->exp_bytes;
    if (cudaMemcpy((void*)L->eptr_dev, ptrs.data(), (size_t)D.E * sizeof(void*), cudaMemcpyHostToDevice) !=
        cudaSuccess)
      return fail(K3MOE_ERR_CUDA, "pointer table upload failed");
  } else {
    k3moe_cache* C = L->cache;
    L->cache = nullptr;
    const int rc = attach_cache(L, C);
    if (rc) return rc;
  }
  L->last_stream = s;
  return K3MOE_OK;
}

uint64_t pool_header_checksum(const k3moe_pool_header* h) {  // FNV-1a 64 over every field before it
  const uint8_t* p = reinterpret_cast<const uint8_t*>(h);
  uint64_t x = 1469598103934665603ull;
  for (size_t i = 0; i < offsetof(k3moe_pool_header, checksum); ++i) x = (x ^ p[i]) * 1099511628211ull;
  return x;
}

}  // namespace

extern "C" {

int k3moe_pack_experts(const k3moe_dims* dims, const void* canon_nib, const void* canon_scale, int src_on_device,
                       const float* W_r, const float* bias, k3moe_cache* cache, void* stream, k3moe_layer** out) {
  if (!out) return fail(K3MOE_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!canon_nib || !canon_scale) return fail(K3MOE_ERR_INVALID_ARG, "NULL input pointer");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  k3moe_layer* L = nullptr;
  int rc = layer_begin(dims, src_on_device, W_r, bias, cache, s, &L);
  if (rc) return rc;
  const k3moe_dims D = *dims;
  const size_t eb = L->exp_bytes;
  auto bail = [&](int code) {
    L->cache = nullptr;
    free_layer(L);
    return code;
  };
  const size_t cn = 3ull * D.f * D.d / 2, cs = 3ull * D.f * D.d / 32;
  // chunk of experts packed per pass: bounded staging (about 2 GB)
  int chunk = (int)std::max<size_t>(1, std::min<size_t>(D.E, (size_t)(2ull << 30) / (cn + cs + eb)));
  uint8_t* stage_nib = nullptr;
  uint8_t* stage_scl = nullptr;
  uint8_t* stage_out = nullptr;
  if ((!src_on_device && (cudaMalloc(&stage_nib, (size_t)chunk * cn) != cudaSuccess ||
                          cudaMalloc(&stage_scl, (size_t)chunk * cs) != cudaSuccess)) ||
      (cache && cudaMalloc(&stage_out, (size_t)chunk * eb) != cudaSuccess)) {
    cudaGetLastError();
    cudaFree(stage_nib);
    cudaFree(stage_scl);
    cudaFree(stage_out);
    return bail(fail(K3MOE_ERR_OOM, "pack staging allocation failed"));
  }
  bool ok = true;
  {
    const int32_t init[4] = {0, 255, 0, 0};  // flags, min scale byte, max scale byte
    ok = cudaMemcpyAsync(L->ws.bad, init, sizeof(init), cudaMemcpyHostToDevice, s) == cudaSuccess &&
         cudaStreamSynchronize(s) == cudaSuccess;
  }
  for (int e0 = 0; e0 < D.E && ok; e0 += chunk) {
    const int n = std::min(chunk, D.E - e0);
    const uint8_t* src_n;
    const uint8_t* src_s;
    if (src_on_device) {
      src_n = (const uint8_t*)canon_nib + (size_t)e0 * cn;
      src_s = (const uint8_t*)canon_scale + (size_t)e0 * cs;
    } else {
      ok = cudaMemcpyAsync(stage_nib, (const uint8_t*)canon_nib + (size_t)e0 * cn, (size_t)n * cn,
                           cudaMemcpyHostToDevice, s) == cudaSuccess &&
           cudaMemcpyAsync(stage_scl, (const uint8_t*)canon_scale + (size_t)e0 * cs, (size_t)n * cs,
                           cudaMemcpyHostToDevice, s) == cudaSuccess;
      src_n = stage_nib;
      src_s = stage_scl;
    }
    uint8_t* dst = cache ? stage_out : L->packed + (size_t)e0 * eb;
    ok = ok && launch_pack(src_n, src_s, n, D.d, D.f, dst, L->ws.bad, s) == cudaSuccess;
    if (ok && cache)
      ok = cudaMemcpyAsync(L->pool + (size_t)e0 * eb, stage_out, (size_t)n * eb, cudaMemcpyDeviceToHost, s) ==
           cudaSuccess;
    if (ok && (!src_on_device || cache)) ok = cudaStreamSynchronize(s) == cudaSuccess;  // staging reused next chunk
  }
  int32_t flags[4] = {0, 255, 0, 0};
  if (ok) ok = cudaMemcpyAsync(flags, L->ws.bad, sizeof(flags), cudaMemcpyDeviceToHost, s) == cudaSuccess;
  if (ok) ok = cudaStreamSynchronize(s) == cudaSuccess;
  cudaFree(stage_nib);
  cudaFree(stage_scl);
  cudaFree(stage_out);
  if (!ok) return bail(fail(K3MOE_ERR_CUDA, "packing failed: %s", cudaGetErrorString(cudaGetLastError())));
  const int32_t bad = flags[0];
  if (bad & 1) return bail(fail(K3MOE_ERR_INVALID_ARG, "a scale byte is 255 (E8M0 NaN)"));
  L->zero_scales = (bad & 2) != 0;
  L->s_min = flags[1];
  L->s_max = flags[2];
  if ((rc = layer_finish(L, s))) return bail(rc);
  *out = L;
  return K3MOE_OK;
}

int k3moe_pool_header_get(k3moe_layer* L, k3moe_pool_header* out) {
  if (!L || !out) return fail(K3MOE_ERR_INVALID_ARG, "NULL argument");
  memset(out, 0, sizeof(*out));
  out->magic = K3MOE_POOL_MAGIC;
  out->version = K3MOE_POOL_VERSION;
  out->d = L->dims.d;
  out->f = L->dims.f;
  out->E = L->dims.E;
  out->s_min = L->s_min;
  out->s_max = L->s_max;
  out->zero_scales = L->zero_scales ? 1 : 0;
  out->expert_bytes = L->exp_bytes;
  out->checksum = pool_header_checksum(out);
  return K3MOE_OK;
}

int k3moe_pool_header_check(const k3moe_pool_header* h, const k3moe_dims* dims) {
  if (!h || !dims) return fail(K3MOE_ERR_INVALID_ARG, "NULL argument");
  int rc = check_dims(dims);
  if (rc) return rc;
  if (h->magic != K3MOE_POOL_MAGIC) return fail(K3MOE_ERR_INVALID_ARG, "not a packed-pool header (magic 0x%08x)", h->magic);
  if (h->version != K3MOE_POOL_VERSION)
    return fail(K3MOE_ERR_INVALID_ARG, "packed-pool layout version %u, this library writes %u", h->version,
                (unsigned)K3MOE_POOL_VERSION);
  if (h->checksum != pool_header_checksum(h)) return fail(K3MOE_ERR_INVALID_ARG, "packed-pool header checksum mismatch");
  if (h->d != dims->d || h->f != dims->f || h->E != dims->E)
    return fail(K3MOE_ERR_INVALID_ARG, "pool holds d=%d f=%d E=%d, dims say d=%d f=%d E=%d", h->d, h->f, h->E, dims->d,
                dims->f, dims->E);
  if (h->expert_bytes != packed_expert_bytes(dims->d, dims->f))
    return fail(K3MOE_ERR_INVALID_ARG, "pool expert size %llu != %zu", (unsigned long long)h->expert_bytes,
                packed_expert_bytes(dims->d, dims->f));
  if (h->s_min < 0 || h->s_max > 254 || h->s_min > h->s_max || (h->zero_scales != 0 && h->zero_scales != 1) ||
      (h->zero_scales == 1) != (h->s_min == 0))
    return fail(K3MOE_ERR_INVALID_ARG, "pool scale range %d..%d (zero flag %d) is not valid", h->s_min, h->s_max,
                h->zero_scales);
  return K3MOE_OK;
}

int k3moe_layer_from_packed(const k3moe_dims* dims, const k3moe_pool_header* header, const void* packed,
                            int src_on_device, const float* W_r, const float* bias, k3moe_cache* cache, void* stream,
                            k3moe_layer** out) {
  if (!out) return fail(K3MOE_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!packed) return fail(K3MOE_ERR_INVALID_ARG, "NULL input pointer");
  int rc = k3moe_pool_header_check(header, dims);
  if (rc) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  k3moe_layer* L = nullptr;
  if ((rc = layer_begin(dims, src_on_device, W_r, bias, cache, s, &L))) return rc;
  const size_t total = (size_t)dims->E * L->exp_bytes;
  cudaError_t e;
  if (!cache)
    e = cudaMemcpyAsync(L->packed, packed, total, src_on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice, s);
  else
    e = cudaMemcpyAsync(L->pool, packed, total, src_on_device ? cudaMemcpyDeviceToHost : cudaMemcpyHostToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    L->cache = nullptr;
    free_layer(L);
    return fail(K3MOE_ERR_CUDA, "packed pool copy failed: %s", cudaGetErrorString(e));
  }
  L->s_min = header->s_min;
  L->s_max = header->s_max;
  L->zero_scales = header->zero_scales != 0;
  if ((rc = layer_finish(L, s))) {
    L->cache = nullptr;
    free_layer(L);
    return rc;
  }
  *out = L;
  return K3MOE_OK;
}

void k3moe_layer_free(k3moe_layer* L) { free_layer(L); }

int k3moe_residual_rmsnorm(const float* y, const void* x, int T, int d, float eps, void* x_next, void* x_norm,
                           void* stream) {
  if (!y || !x || !x_next || !x_norm) return fail(K3MOE_ERR_INVALID_ARG, "NULL argument");
  if (!aligned_to(y, 4) || !aligned_to(x, 2) || !aligned_to(x_next, 2) || !aligned_to(x_norm, 2))
    return fail(K3MOE_ERR_INVALID_ARG, "y must be 4-byte and x, x_next, x_norm 2-byte aligned");
  if (T < 1 || d < 1 || d > 65536) return fail(K3MOE_ERR_INVALID_ARG, "T=%d, d=%d out of range", T, d);
  if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(K3MOE_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if (x_norm == x_next) return fail(K3MOE_ERR_INVALID_ARG, "x_norm must not alias x_next");
  CUDA_TRY(launch_residual_rmsnorm(y, reinterpret_cast<const uint16_t*>(x), T, d, eps,
                                   reinterpret_cast<uint16_t*>(x_next), reinterpret_cast<uint16_t*>(x_norm),
                                   reinterpret_cast<cudaStream_t>(stream)));
  return K3MOE_OK;
}

int k3moe_layer_set_cache(k3moe_layer* L, k3moe_cache* C) {
  if (!L || !C) return fail(K3MOE_ERR_INVALID_ARG, "NULL argument");
  if (!L->pool) return fail(K3MOE_ERR_INVALID_ARG, "layer was packed without a cache (its experts live on the device)");
  if (C->slot_bytes != L->exp_bytes)
    return fail(K3MOE_ERR_INVALID_ARG, "cache slot_bytes %zu != packed expert bytes %zu", C->slot_bytes, L->exp_bytes);
  if (C == L->cache) return K3MOE_OK;
  if (L->last_stream) CUDA_TRY(cudaStreamSynchronize(L->last_stream));
  if (L->cache) CUDA_TRY(cudaStreamSynchronize(L->cache->copy_stream));
  if (C->device_lru) {
    const long long need = std::min<long long>(L->dims.E, (long long)L->dims.T_max * L->dims.k);
    if (need > C->n_slots)
      return fail(K3MOE_ERR_BUDGET_TOO_SMALL, "a call may need %lld experts resident, the cache has %d slots", need,
                  C->n_slots);
  }
  detach_cache(L);
  return attach_cache(L, C);
}

int k3moe_router_topk(k3moe_layer* L, const void* x, int T, int32_t* idx, float* w, void* stream) {
  if (!L || !x || !idx || !w) return fail(K3MOE_ERR_INVALID_ARG, "NULL argument");
  if ((reinterpret_cast<uintptr_t>(x) & 15u) != 0) return fail(K3MOE_ERR_INVALID_ARG, "x must be 16-byte aligned");
  if (!aligned_to(idx, 4) || !aligned_to(w, 4)) return fail(K3MOE_ERR_INVALID_ARG, "idx and w must be 4-byte aligned");
  if (T < 1 || T > L->dims.T_max) return fail(K3MOE_ERR_INVALID_ARG, "T=%d must be in 1..%d", T, L->dims.T_max);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  L->last_stream = s;
  int rc = run_routing(L, x, T, s, false);
  if (rc) return rc;
  const size_t n = (size_t)T * L->dims.k;
  CUDA_TRY(cudaMemcpyAsync(idx, L->ws.idx, n * 4, cudaMemcpyDeviceToDevice, s));
  CUDA_TRY(cudaMemcpyAsync(w, L->ws.w, n * 4, cudaMemcpyDeviceToDevice, s));
  return K3MOE_OK;
}

int k3moe_bucket(k3moe_layer* L, const int32_t* idx, int T, int32_t* counts, int32_t* offsets, int32_t* perm,
                 void* stream) {
  if (!L || !idx || !counts || !offsets || !perm) return fail(K3MOE_ERR_INVALID_ARG, "NULL argument");
  if (!aligned_to(idx, 4) || !aligned_to(counts, 4) || !aligned_to(offsets, 4) || !aligned_to(perm, 4))
    return fail(K3MOE_ERR_INVALID_ARG, "idx, counts, offsets and perm must be 4-byte aligned");
  if (T < 1 || T > L->dims.T_max) return fail(K3MOE_ERR_INVALID_ARG, "T=%d must be in 1..%d", T, L->dims.T_max);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  L->last_stream = s;
  const k3moe_dims& D = L->dims;
  return timed_launch(L, KID_BUCKET, s, [&] {
    return launch_bucket(idx, T, D.k, D.E, counts, offsets, perm, L->ws.act, L->ws.nact, L->ws.units, L->ws.nunits,
                         L->ws.w, L->ws.xscale, L->ws.chist, s, false);  // the caller gets counts, offsets and perm
  });
}

int k3moe_layer_forward(k3moe_layer* L, const void* x, int T, float* y, void* stream) {
  if (!L || !x || !y) return fail(K3MOE_ERR_INVALID_ARG, "NULL argument");
  if ((reinterpret_cast<uintptr_t>(x) & 15u) != 0) return fail(K3MOE_ERR_INVALID_ARG, "x must be 16-byte aligned");
  // the combine writes y four floats at a time
  if ((reinterpret_cast<uintptr_t>(y) & 15u) != 0) return fail(K3MOE_ERR_INVALID_ARG, "y must be 16-byte aligned");
  if (T < 1 || T > L->dims.T_max) return fail(K3MOE_ERR_INVALID_ARG, "T=%d must be in 1..%d", T, L->dims.T_max);
  return forward_impl(L, x, T, y, reinterpret_cast<cudaStream_t>(stream));
}

int k3moe_layer_forward_host(k3moe_layer* L, const void* x_host, int T, float* y_host, void* stream) {
  if (!L || !x_host || !y_host) return fail(K3MOE_ERR_INVALID_ARG, "NULL argument");
  if (T < 1 || T > L->dims.T_max) return fail(K3MOE_ERR_INVALID_ARG, "T=%d must be in 1..%d", T, L->dims.T_max);
  const k3moe_dims& D = L->dims;
  if (!L->x_stage) {
    if (cudaMalloc(&L->x_stage, (size_t)D.T_max * D.d * 2) != cudaSuccess ||
        cudaMalloc(&L->y_stage, (size_t)D.T_max * D.d * 4) != cudaSuccess ||
        cudaHostAlloc((void**)&L->flags_host, 16, cudaHostAllocDefault) != cudaSuccess) {
      cudaGetLastError();
      return fail(K3MOE_ERR_OOM, "host-forward staging allocation failed");
    }
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  CUDA_TRY(cudaMemcpyAsync(L->x_stage, x_host, (size_t)T * D.d * 2, cudaMemcpyHostToDevice, s));
  int rc = forward_impl(L, L->x_stage, T, L->y_stage, s);
  if (rc) return rc;
  CUDA_TRY(cudaMemcpyAsync(y_host, L->y_stage, (size_t)T * D.d * 4, cudaMemcpyDeviceToHost, s));
  // the error flags come back on the same stream, so one synchronisation covers both copies
  CUDA_TRY(cudaMemcpyAsync(L->flags_host, L->ws.sync + 1, 4, cudaMemcpyDeviceToHost, s));
  CUDA_TRY(cudaStreamSynchronize(s));
  const uint32_t flags = *reinterpret_cast<volatile uint32_t*>(L->flags_host);
  if (flags) {
    CUDA_TRY(reset_after_timeout(L));
    return fail(K3MOE_ERR_TIMEOUT, "a device-side wait gave up (flags 0x%x)", flags);
  }
  return K3MOE_OK;
}

int k3moe_graph_create(k3moe_layer* L, const void* x, int T, int calls, float* y, void* stream, k3moe_graph** out) {
  if (!out) return fail(K3MOE_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!L || !x || !y) return fail(K3MOE_ERR_INVALID_ARG, "NULL argument");
  if (calls < 1) return fail(K3MOE_ERR_INVALID_ARG, "calls=%d must be at least 1", calls);
  if (T < 1 || T > L->dims.T_max) return fail(K3MOE_ERR_INVALID_ARG, "T=%d must be in 1..%d", T, L->dims.T_max);
  if ((reinterpret_cast<uintptr_t>(x) & 15u) != 0 || (reinterpret_cast<uintptr_t>(y) & 15u) != 0)
    return fail(K3MOE_ERR_INVALID_ARG, "x and y must be 16-byte aligned");
  if (L->cache)
    return fail(K3MOE_ERR_UNSUPPORTED, "a cache-mode layer's calls synchronise the host and cannot be captured");
  if (L->profiling) return fail(K3MOE_ERR_INVALID_ARG, "per-kernel timing is on: turn k3moe_profile off to capture");
  const size_t xs = (size_t)T * L->dims.d * 2;  // bytes of one call's x
  const size_t ys = (size_t)T * L->dims.d;      // floats of one call's y
  const uint8_t* xb = static_cast<const uint8_t*>(x);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // eager once: checks the calls and sets every kernel's launch attributes outside the capture
  for (int c = 0; c < calls; ++c) {
    const int rc = forward_impl(L, xb + c * xs, T, y + c * ys, s);
    if (rc) return rc;
  }
  // capture on a private stream (the caller's may be the legacy stream, which cannot capture)
  cudaStream_t cs = nullptr;
  CUDA_TRY(cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking));
  cudaError_t e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
  int rc = K3MOE_OK;
  for (int c = 0; c < calls && e == cudaSuccess && rc == K3MOE_OK; ++c) rc = forward_impl(L, xb + c * xs, T, y + c * ys, cs);
  cudaGraph_t g = nullptr;
  const cudaError_t e2 = e == cudaSuccess ? cudaStreamEndCapture(cs, &g) : e;
  L->last_stream = s;
  cudaStreamDestroy(cs);
  if (rc != K3MOE_OK || e2 != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    cudaGetLastError();
    return rc != K3MOE_OK ? rc : fail(K3MOE_ERR_CUDA, "capturing the layer calls failed: %s", cudaGetErrorString(e2));
  }
  cudaGraphExec_t ex = nullptr;
  e = cudaGraphInstantiate(&ex, g, 0);
  if (e != cudaSuccess) {
    cudaGraphDestroy(g);
    cudaGetLastError();
    return fail(K3MOE_ERR_CUDA, "instantiating the captured calls failed: %s", cudaGetErrorString(e));
  }
  *out = new k3moe_graph{L, g, ex};
  return K3MOE_OK;
}

int k3moe_graph_launch(k3moe_graph* G, void* stream) {
  if (!G) return fail(K3MOE_ERR_INVALID_ARG, "graph is NULL");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  G->layer->last_stream = s;  // k3moe_sync waits for the replay here
  CUDA_TRY(cudaGraphLaunch(G->exec, s));
  return K3MOE_OK;
}

void k3moe_graph_destroy(k3moe_graph* G) {
  if (!G) return;
  if (G->exec) cudaGraphExecDestroy(G->exec);
  if (G->graph) cudaGraphDestroy(G->graph);
  delete G;
}

int k3moe_sync(k3moe_layer* L) {
  if (!L) return fail(K3MOE_ERR_INVALID_ARG, "layer is NULL");
  if (L->last_stream) CUDA_TRY(cudaStreamSynchronize(L->last_stream));
  CUDA_TRY(cudaDeviceSynchronize());
  if (L->cache) {
    // every call and copy so far has finished: a prefetch may take any slot
    L->cache->done_before = L->cache->calls_issued;
    L->cache->fast_since_sync = false;
    L->cache->prefetch_pending = false;
  }
  uint32_t flags = 0;
  CUDA_TRY(cudaMemcpy(&flags, L->ws.sync + 1, 4, cudaMemcpyDeviceToHost));
  if (flags) {
    CUDA_TRY(reset_after_timeout(L));
    return fail(K3MOE_ERR_TIMEOUT, "a device-side wait gave up (flags 0x%x); the results of the calls since the "
                "last k3moe_sync are invalid", flags);
  }
  return K3MOE_OK;
}

int k3moe_set_option(k3moe_layer* L, int option, long long value) {
  if (!L) return fail(K3MOE_ERR_INVALID_ARG, "layer is NULL");
  switch (option) {
    case K3MOE_OPT_DEVICE_WAIT_NS:
      if (value < 1000000 || value > 60000000000LL)
        return fail(K3MOE_ERR_INVALID_ARG, "DEVICE_WAIT_NS must be in 1e6..6e10");
      L->wait_ns = (unsigned long long)value;
      return K3MOE_OK;
    case K3MOE_OPT_RING_DEPTH:
      if (value < 0 || value > 6) return fail(K3MOE_ERR_INVALID_ARG, "RING_DEPTH must be in 0..6");
      L->ring_depth = (int)value;
      return K3MOE_OK;
    case K3MOE_OPT_TEST_FAIL_COPY:
      if (value < 0 || value > (1LL << 30)) return fail(K3MOE_ERR_INVALID_ARG, "TEST_FAIL_COPY must be in 0..2^30");
      L->test_fail_copy = (int)value;
      return K3MOE_OK;
    case K3MOE_OPT_TEST_STALL:
      if (value != 0 && value != 1) return fail(K3MOE_ERR_INVALID_ARG, "TEST_STALL must be 0 or 1");
      L->test_stall = (int)value;
      return K3MOE_OK;
    case K3MOE_OPT_PATH:
      if (value != K3MOE_PATH_AUTO && value != K3MOE_PATH_DECODE && value != K3MOE_PATH_GEMM)
        return fail(K3MOE_ERR_INVALID_ARG, "unknown path %lld", value);
      L->path = (int)value;
      return K3MOE_OK;
    case K3MOE_OPT_MISS_PATH:
      if (value != K3MOE_MISS_COPY_ENGINE && value != K3MOE_MISS_ZERO_COPY)
        return fail(K3MOE_ERR_INVALID_ARG, "unknown miss path %lld", value);
      L->miss_path = (int)value;
      return K3MOE_OK;
    case K3MOE_OPT_ACTIVATION:
      if (value != K3MOE_ACT_SWIGLU && value != K3MOE_ACT_SITU_GLU)
        return fail(K3MOE_ERR_INVALID_ARG, "unknown activation %lld", value);
      L->activation = (int)value;
      return K3MOE_OK;
    case K3MOE_OPT_GEMM_MIN_T:
      if (value < 1) return fail(K3MOE_ERR_INVALID_ARG, "GEMM_MIN_T must be >= 1");
      L->gemm_min_t = value;
      return K3MOE_OK;
    default:
      return fail(K3MOE_ERR_INVALID_ARG, "unknown option %d", option);
  }
}

int k3moe_profile(k3moe_layer* L, int enable) {
  if (!L) return fail(K3MOE_ERR_INVALID_ARG, "layer is NULL");
  if (L->last_stream) cudaStreamSynchronize(L->last_stream);
  for (auto& t : L->timed) {
    L->spare_events.push_back(t.a);
    L->spare_events.push_back(t.b);
  }
  L->timed.clear();
  for (int i = 0; i < K3MOE_K_COUNT; ++i) {
    L->prof_ms[i] = 0;
    L->prof_n[i] = 0;
  }
  L->profiling = enable != 0;
  return K3MOE_OK;
}

int k3moe_profile_read(k3moe_layer* L, k3moe_kernel_time* out) {
  if (!L || !out) return fail(K3MOE_ERR_INVALID_ARG, "NULL argument");
  for (auto& t : L->timed) {
    float ms = 0.f;
    CUDA_TRY(cudaEventSynchronize(t.b));
    CUDA_TRY(cudaEventElapsedTime(&ms, t.a, t.b));
    L->prof_ms[t.kid] += ms;
    L->prof_n[t.kid] += 1;
    L->spare_events.push_back(t.a);
    L->spare_events.push_back(t.b);
  }
  L->timed.clear();
  for (int i = 0; i < K3MOE_K_COUNT; ++i) {
    out[i].ms_total = L->prof_ms[i];
    out[i].launches = L->prof_n[i];
  }
  return K3MOE_OK;
}

int k3moe_debug_buffer(k3moe_layer* L, int which, void** dev_ptr, size_t* bytes) {
  if (!L || !dev_ptr || !bytes) return fail(K3MOE_ERR_INVALID_ARG, "NULL argument");
  const k3moe_dims& D = L->dims;
  const size_t P = (size_t)D.T_max * D.k;
  switch (which) {
    case 0: *dev_ptr = L->ws.hbuf; *bytes = P * D.f * 4; return K3MOE_OK;
    case 1: *dev_ptr = L->ws.obuf; *bytes = P * D.d * 4; return K3MOE_OK;
    case 2: *dev_ptr = L->ws.idx; *bytes = P * 4; return K3MOE_OK;
    default: return fail(K3MOE_ERR_INVALID_ARG, "unknown buffer %d", which);
  }
}

int k3moe_read_packed(k3moe_layer* L, int e, void* dst) {
  if (!L || !dst) return fail(K3MOE_ERR_INVALID_ARG, "NULL argument");
  if (e < 0 || e >= L->dims.E) return fail(K3MOE_ERR_INVALID_ARG, "expert %d out of range", e);
  if (L->cache) {
    memcpy(dst, L->pool + (size_t)e * L->exp_bytes, L->exp_bytes);
    return K3MOE_OK;
  }
  if (L->last_stream) CUDA_TRY(cudaStreamSynchronize(L->last_stream));
  CUDA_TRY(cudaMemcpy(dst, L->packed + (size_t)e * L->exp_bytes, L->exp_bytes, cudaMemcpyDeviceToHost));
  return K3MOE_OK;
}

}  // extern "C"
