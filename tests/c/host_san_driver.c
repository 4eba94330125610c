/* The library's host code under AddressSanitizer and UndefinedBehaviorSanitizer: this plain C
 * program is compiled with -fsanitize=address,undefined and linked to libk3moe_san.so (the
 * library with its host code built the same way).  Any invalid memory access, leak of a
 * deleted object's fields or undefined behaviour in the argument checks, the cache simulator or
 * the expert cache's LRU bookkeeping aborts the run.
 *   Without a GPU: the cache simulator on random traces under every policy, and the refusals.
 *   With a GPU: also a layer in cache mode driven through the host-buffer entry point, with
 *   prefetches between the calls (hits,
 *   misses, evictions, a failed copy injected on the host, a move to another cache).
 * Prints "ok cpu" (no device) or "ok gpu", exit code 0, when every check holds. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "k3moe.h"

#define CHECK(cond, code)                                    \
  do {                                                       \
    if (!(cond)) {                                           \
      fprintf(stderr, "check %d failed: %s (%s)\n", code, #cond, k3moe_last_error()); \
      return code;                                           \
    }                                                        \
  } while (0)

static uint64_t g_state = 0x9E3779B97F4A7C15ull;
static uint64_t rnd(void) { /* xorshift64 */
  g_state ^= g_state << 13;
  g_state ^= g_state >> 7;
  g_state ^= g_state << 17;
  return g_state;
}

static int simulator_checks(void) {
  enum { kCalls = 3000, kKeys = 256, kMaxPer = 16 };
  int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * kCalls * kMaxPer);
  int64_t* starts = (int64_t*)malloc(sizeof(int64_t) * (kCalls + 1));
  int n = 0;
  starts[0] = 0;
  for (int c = 0; c < kCalls; ++c) {
    const int m = 1 + (int)(rnd() % kMaxPer);
    for (int i = 0; i < m; ++i) {
      int64_t kk;
      int dup;
      do { /* distinct within the call */
        kk = (int64_t)(rnd() % kKeys);
        dup = 0;
        for (int j = (int)starts[c]; j < n; ++j) dup |= keys[j] == kk;
      } while (dup);
      keys[n++] = kk;
    }
    starts[c + 1] = n;
  }
  const int policies[3] = {K3MOE_POLICY_LRU, K3MOE_POLICY_MIN, K3MOE_POLICY_RANDOM};
  for (int slots = kMaxPer; slots <= 64; slots += 24)
    for (int p = 0; p < 3; ++p) {
      k3moe_cache_sim_stats st;
      CHECK(k3moe_cache_simulate(keys, starts, kCalls, slots, policies[p], 7, &st) == K3MOE_OK, 100 + p);
      CHECK(st.hits + st.misses == n, 110 + p);
      CHECK(st.evictions <= st.misses && st.misses >= slots, 120 + p);  /* every key set spans > slots keys */
    }
  k3moe_cache_sim_stats st;
  int biggest = 0; /* a call of kMaxPer keys exists in 3000 draws; with kMaxPer - 1 slots it cannot fit */
  for (int c = 0; c < kCalls; ++c) biggest = (int)(starts[c + 1] - starts[c]) > biggest ? (int)(starts[c + 1] - starts[c]) : biggest;
  CHECK(biggest == kMaxPer, 129);
  CHECK(k3moe_cache_simulate(keys, starts, kCalls, kMaxPer - 1, K3MOE_POLICY_LRU, 0, &st) == K3MOE_ERR_BUDGET_TOO_SMALL,
        130);
  keys[1] = keys[0];
  starts[1] = 2; /* call 0 = keys[0], keys[1]: a repeated key */
  CHECK(k3moe_cache_simulate(keys, starts, 1, 8, K3MOE_POLICY_MIN, 0, &st) == K3MOE_ERR_INVALID_ARG, 131);
  starts[1] = -1;
  CHECK(k3moe_cache_simulate(keys, starts, 1, 8, K3MOE_POLICY_LRU, 0, &st) == K3MOE_ERR_INVALID_ARG, 132);
  CHECK(k3moe_cache_simulate(keys, starts, 1, 8, 99, 0, &st) == K3MOE_ERR_INVALID_ARG, 133);
  free(keys);
  free(starts);
  return 0;
}

static int refusal_checks(void) {
  const k3moe_dims bad = {100, 1536, 896, 16, 1};
  const k3moe_dims ok = {256, 128, 8, 2, 2};
  k3moe_layer* layer = NULL;
  const float w[4] = {0};
  CHECK(k3moe_pack_experts(&bad, w, w, 0, w, NULL, NULL, NULL, &layer) == K3MOE_ERR_INVALID_ARG, 200);
  CHECK(k3moe_pack_experts(&ok, NULL, w, 0, w, NULL, NULL, NULL, &layer) == K3MOE_ERR_INVALID_ARG, 201);
  CHECK(k3moe_pack_experts(&ok, w, w, 2, w, NULL, NULL, NULL, &layer) == K3MOE_ERR_INVALID_ARG, 202);
  CHECK(layer == NULL, 203);
  k3moe_cache* cache = NULL;
  CHECK(k3moe_cache_create(100, 256, &cache) == K3MOE_ERR_INVALID_ARG, 204);
  CHECK(k3moe_cache_create(1 << 20, 100, &cache) == K3MOE_ERR_INVALID_ARG, 205);
  CHECK(k3moe_set_option(NULL, K3MOE_OPT_PATH, 0) == K3MOE_ERR_INVALID_ARG, 206);
  CHECK(k3moe_residual_rmsnorm(NULL, w, 1, 4, 1e-6f, (void*)w, (void*)w, NULL) == K3MOE_ERR_INVALID_ARG, 207);
  CHECK(k3moe_router_topk_noalloc(NULL, w, NULL, 1, 4, 8, 2, NULL, NULL, NULL) == K3MOE_ERR_INVALID_ARG, 208);
  CHECK(k3moe_router_topk_noalloc(w, w, NULL, 17, 256, 4096, 4, (int32_t*)w, (float*)w, NULL) ==
            K3MOE_ERR_INVALID_ARG, 209);
  k3moe_layer_free(NULL);
  k3moe_cache_destroy(NULL);
  CHECK(strlen(k3moe_last_error()) > 0, 210);
  return 0;
}

/* A tiny layer (d=256, f=128, E=8, k=2) in cache mode, experts brought in through 6 slots. */
static int gpu_checks(void) {
  const k3moe_dims dm = {256, 128, 8, 2, 2};
  const size_t eb = k3moe_packed_expert_bytes(&dm);
  k3moe_cache *c1 = NULL, *c2 = NULL;
  if (k3moe_cache_create(6 * eb, eb, &c1) != K3MOE_OK) return -1; /* no device */
  CHECK(k3moe_cache_create(8 * eb, eb, &c2) == K3MOE_OK, 300);
  const size_t nb = (size_t)3 * dm.f * dm.d / 2, sb = (size_t)3 * dm.f * dm.d / 32;
  uint8_t* nib = (uint8_t*)malloc(nb * dm.E);
  uint8_t* scl = (uint8_t*)malloc(sb * dm.E);
  float* wr = (float*)malloc(sizeof(float) * dm.E * dm.d);
  for (size_t i = 0; i < nb * dm.E; ++i) nib[i] = (uint8_t)rnd();
  for (size_t i = 0; i < sb * dm.E; ++i) scl[i] = (uint8_t)(121 + rnd() % 5);
  for (int i = 0; i < dm.E * dm.d; ++i) wr[i] = (float)((int)(rnd() % 2001) - 1000) * 1e-4f;
  k3moe_layer* layer = NULL;
  CHECK(k3moe_pack_experts(&dm, nib, scl, 0, wr, NULL, c1, NULL, &layer) == K3MOE_OK, 301);
  uint16_t x[2 * 256];
  float y[2 * 256];
  int failed = 0;
  for (int call = 0; call < 40; ++call) {
    for (int i = 0; i < 2 * 256; ++i) x[i] = (uint16_t)(0x3c00u + (rnd() % 0x0400u) + ((rnd() & 1u) << 15));
    if (call == 20) CHECK(k3moe_set_option(layer, K3MOE_OPT_TEST_FAIL_COPY, 1) == K3MOE_OK, 302);
    if ((call & 1) && call < 30) { /* prefetch three experts (repeats allowed) before the call */
      int32_t ids[3];
      for (int j = 0; j < 3; ++j) ids[j] = (int32_t)(rnd() % (uint32_t)dm.E);
      int got = -1;
      const int prc = k3moe_cache_prefetch(layer, ids, 3, &got);
      if (prc == K3MOE_ERR_CUDA && call >= 20 && !failed)
        failed = 1; /* the injected copy failure came in a prefetch */
      else
        CHECK(prc == K3MOE_OK && got >= 0 && got <= 3, 309);
    }
    const int rc = k3moe_layer_forward_host(layer, x, 2, y, NULL);
    if (rc == K3MOE_ERR_CUDA && call >= 20 && !failed) {
      failed = 1; /* the injected copy failure (a call that needed a copy) */
      continue;
    }
    CHECK(rc == K3MOE_OK, 303);
    if (call == 30) CHECK(k3moe_layer_set_cache(layer, c2) == K3MOE_OK, 304);
  }
  CHECK(failed, 305);
  k3moe_cache_stats_t st1, st2;
  CHECK(k3moe_cache_stats(c1, &st1) == K3MOE_OK && k3moe_cache_stats(c2, &st2) == K3MOE_OK, 306);
  CHECK(st1.misses > 0 && st1.evictions > 0 && st2.misses > 0, 307);
  CHECK(st1.prefetched > 0 && st1.h2d_bytes == (st1.misses + st1.prefetched) * eb, 310);
  int32_t bad = dm.E;
  CHECK(k3moe_cache_prefetch(layer, &bad, 1, NULL) == K3MOE_ERR_INVALID_ARG, 311);
  CHECK(k3moe_cache_reset_stats(c2) == K3MOE_OK, 308);
  k3moe_layer_free(layer);
  k3moe_cache_destroy(c1);
  k3moe_cache_destroy(c2);
  free(nib);
  free(scl);
  free(wr);
  return 0;
}

int main(void) {
  int rc = simulator_checks();
  if (rc) return rc;
  rc = refusal_checks();
  if (rc) return rc;
  rc = gpu_checks();
  if (rc > 0) return rc;
  puts(rc < 0 ? "ok cpu" : "ok gpu");
  return 0;
}
