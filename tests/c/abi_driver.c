/* A plain C caller of the library, compiled with a C compiler against include/k3moe.h and linked
 * to libk3moe.so: the boundary is usable without Python or C++.  It touches no GPU: it checks the
 * packed-size rule, the host-only cache-policy simulator (the textbook reference string: 3 frames,
 * OPT 9 faults, LRU 12) and that bad arguments are refused with an error code and a message
 * before any device work.  Exit code 0 and "ok" on stdout when every check holds. */
#include <stdio.h>
#include <string.h>

#include "k3moe.h"

#define CHECK(cond, code)                              \
  do {                                                 \
    if (!(cond)) {                                     \
      fprintf(stderr, "check %d failed: %s\n", code, #cond); \
      return code;                                     \
    }                                                  \
  } while (0)

int main(void) {
  const k3moe_dims k3 = {7168, 1536, 896, 16, 1};
  const k3moe_dims bad = {100, 1536, 896, 16, 1}; /* d not a multiple of 128 */
  CHECK(k3moe_packed_expert_bytes(&k3) == 17547264u, 1);
  CHECK(k3moe_packed_expert_bytes(&bad) == 0, 2);

  const int64_t ref[20] = {7, 0, 1, 2, 0, 3, 0, 4, 2, 3, 0, 3, 2, 1, 2, 0, 1, 7, 0, 1};
  int64_t starts[21];
  for (int i = 0; i <= 20; ++i) starts[i] = i;
  k3moe_cache_sim_stats st;
  CHECK(k3moe_cache_simulate(ref, starts, 20, 3, K3MOE_POLICY_MIN, 0, &st) == K3MOE_OK, 3);
  CHECK(st.misses == 9 && st.hits == 11 && st.evictions == 6, 4);
  CHECK(k3moe_cache_simulate(ref, starts, 20, 3, K3MOE_POLICY_LRU, 0, &st) == K3MOE_OK, 5);
  CHECK(st.misses == 12 && st.hits == 8 && st.evictions == 9, 6);

  k3moe_layer* layer = NULL;
  const float w[4] = {0};
  CHECK(k3moe_pack_experts(&bad, w, w, 0, w, NULL, NULL, NULL, &layer) == K3MOE_ERR_INVALID_ARG, 7);
  CHECK(layer == NULL, 8);
  const char* msg = k3moe_last_error();
  CHECK(msg != NULL && strstr(msg, "d=100") != NULL, 9);
  CHECK(k3moe_cache_simulate(ref, starts, 20, 0, K3MOE_POLICY_LRU, 0, &st) == K3MOE_ERR_INVALID_ARG, 10);
  CHECK(k3moe_router_topk(NULL, w, 1, NULL, NULL, NULL) == K3MOE_ERR_INVALID_ARG, 11);
  int fetched = -1;
  const int32_t ids[2] = {0, 1};
  CHECK(k3moe_cache_prefetch(NULL, ids, 2, &fetched) == K3MOE_ERR_INVALID_ARG && fetched == 0, 12);
  k3moe_graph* graph = (k3moe_graph*)&fetched; /* must be cleared on refusal */
  CHECK(k3moe_graph_create(NULL, w, 1, 1, (float*)w, NULL, &graph) == K3MOE_ERR_INVALID_ARG && graph == NULL, 13);
  CHECK(k3moe_graph_launch(NULL, NULL) == K3MOE_ERR_INVALID_ARG, 14);
  k3moe_graph_destroy(NULL);
  k3moe_layer_free(NULL);
  puts("ok");
  return 0;
}
