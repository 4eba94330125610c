// cachesim.cu -- replay of an expert-access trace through a cache of expert slots (host only).
//
// "kimi-k3-in-c deep dive", "four reductions", expert LRU paragraph, and its cache-hit figures
// (measured there with a simulator on a recorded routing trace): the engine keeps the most
// recently used experts in RAM and reloads the rest.  This replays a trace of layer calls -- each
// call the set of experts it needs resident at once -- through n_slots expert slots under three
// replacement policies:
//   LRU     the device cache's policy: a call's hits are touched first (in the given order),
//           then each miss takes the least recently used slot not touched by the call;
//   MIN     Belady's offline optimum: a miss in a full cache evicts the resident expert, not
//           needed by the current call, whose next use lies farthest ahead (never used again
//           counts as farthest; ties go to the larger key);
//   RANDOM  a miss in a full cache evicts a uniformly drawn resident expert not needed by the
//           current call (splitmix64 stream from the seed).
// Empty slots are filled before anything is evicted; filling an empty slot is a miss but not an
// eviction.
#include <cstdint>
#include <list>
#include <queue>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "k3moe_internal.cuh"

namespace {

int sim_fail(int code, const char* msg) {
  k3::set_last_error(msg);
  return code;
}

uint64_t splitmix64(uint64_t& state) {
  uint64_t z = (state += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

}  // namespace

extern "C" int k3moe_cache_simulate(const int64_t* keys, const int64_t* call_start, int n_calls, int n_slots,
                                    int policy, unsigned long long seed, k3moe_cache_sim_stats* out) {
  if (!out) return sim_fail(K3MOE_ERR_INVALID_ARG, "cache_simulate: out is NULL");
  if (n_calls < 0 || n_slots < 1) return sim_fail(K3MOE_ERR_INVALID_ARG, "cache_simulate: n_calls < 0 or n_slots < 1");
  if (policy != K3MOE_POLICY_LRU && policy != K3MOE_POLICY_MIN && policy != K3MOE_POLICY_RANDOM)
    return sim_fail(K3MOE_ERR_INVALID_ARG, "cache_simulate: unknown policy");
  if (n_calls > 0 && (!keys || !call_start)) return sim_fail(K3MOE_ERR_INVALID_ARG, "cache_simulate: NULL trace");
  k3moe_cache_sim_stats st{0, 0, 0};
  if (n_calls == 0) {
    *out = st;
    return K3MOE_OK;
  }
  if (call_start[0] != 0) return sim_fail(K3MOE_ERR_INVALID_ARG, "cache_simulate: call_start[0] != 0");
  for (int c = 0; c < n_calls; ++c) {
    if (call_start[c + 1] < call_start[c]) return sim_fail(K3MOE_ERR_INVALID_ARG, "cache_simulate: call_start decreases");
    if (call_start[c + 1] - call_start[c] > n_slots)
      return sim_fail(K3MOE_ERR_BUDGET_TOO_SMALL, "cache_simulate: a call needs more experts than there are slots");
    std::unordered_set<int64_t> seen;
    for (int64_t i = call_start[c]; i < call_start[c + 1]; ++i)
      if (!seen.insert(keys[i]).second)
        return sim_fail(K3MOE_ERR_INVALID_ARG, "cache_simulate: a key repeats within one call");
  }
  const int64_t n = call_start[n_calls];

  if (policy == K3MOE_POLICY_LRU) {
    std::list<int64_t> order;  // front = most recently used
    std::unordered_map<int64_t, std::list<int64_t>::iterator> pos;
    std::vector<int64_t> miss;
    for (int c = 0; c < n_calls; ++c) {
      miss.clear();
      for (int64_t i = call_start[c]; i < call_start[c + 1]; ++i) {
        auto it = pos.find(keys[i]);
        if (it != pos.end()) {
          order.splice(order.begin(), order, it->second);
          ++st.hits;
        } else {
          miss.push_back(keys[i]);
        }
      }
      for (int64_t key : miss) {
        if ((int)order.size() == n_slots) {
          pos.erase(order.back());
          order.pop_back();
          ++st.evictions;
        }
        order.push_front(key);
        pos[key] = order.begin();
        ++st.misses;
      }
    }
  } else if (policy == K3MOE_POLICY_MIN) {
    // next_use[i]: the next call after occurrence i's call that needs the same key (n_calls: never)
    std::vector<int> call_of(n);
    for (int c = 0; c < n_calls; ++c)
      for (int64_t i = call_start[c]; i < call_start[c + 1]; ++i) call_of[i] = c;
    std::vector<int> next_use(n, n_calls);
    std::unordered_map<int64_t, int> later;  // key -> the nearest later call seen so far
    for (int64_t i = n - 1; i >= 0; --i) {
      auto it = later.find(keys[i]);
      next_use[i] = it == later.end() ? n_calls : it->second;
      later[keys[i]] = call_of[i];
    }
    std::unordered_map<int64_t, int> resident;  // key -> its current next use
    std::priority_queue<std::pair<int, int64_t>> heap;  // (next use, key); stale entries skipped
    std::vector<int64_t> miss;
    std::vector<std::pair<int, int64_t>> held;
    std::unordered_set<int64_t> current;
    for (int c = 0; c < n_calls; ++c) {
      miss.clear();
      current.clear();
      for (int64_t i = call_start[c]; i < call_start[c + 1]; ++i) {
        current.insert(keys[i]);
        auto it = resident.find(keys[i]);
        if (it != resident.end()) {
          it->second = next_use[i];
          heap.push({next_use[i], keys[i]});
          ++st.hits;
        } else {
          miss.push_back(keys[i]);
        }
      }
      int64_t mi = 0;
      for (int64_t i = call_start[c]; i < call_start[c + 1]; ++i) {
        if (mi < (int64_t)miss.size() && keys[i] == miss[mi]) {
          if ((int)resident.size() == n_slots) {
            held.clear();
            for (;;) {
              const auto top = heap.top();
              heap.pop();
              auto r = resident.find(top.second);
              if (r == resident.end() || r->second != top.first) continue;  // stale
              if (current.count(top.second)) {
                held.push_back(top);
                continue;
              }
              resident.erase(r);
              ++st.evictions;
              break;
            }
            for (const auto& h : held) heap.push(h);
          }
          resident[keys[i]] = next_use[i];
          heap.push({next_use[i], keys[i]});
          ++st.misses;
          ++mi;
        }
      }
    }
  } else {
    uint64_t rng = seed;
    std::vector<int64_t> slots;               // resident keys
    std::unordered_map<int64_t, size_t> at;   // key -> index in slots
    std::unordered_set<int64_t> current;
    std::vector<int64_t> miss;
    for (int c = 0; c < n_calls; ++c) {
      miss.clear();
      current.clear();
      for (int64_t i = call_start[c]; i < call_start[c + 1]; ++i) {
        current.insert(keys[i]);
        if (at.count(keys[i])) ++st.hits; else miss.push_back(keys[i]);
      }
      for (int64_t key : miss) {
        if ((int)slots.size() == n_slots) {
          // a call needs at most n_slots experts, so some resident one is not needed by it
          size_t v = 0;
          for (;;) {
            v = (size_t)(splitmix64(rng) % (uint64_t)slots.size());
            if (!current.count(slots[v])) break;
          }
          at.erase(slots[v]);
          slots[v] = slots.back();
          slots.pop_back();
          if (v < slots.size()) at[slots[v]] = v;
          ++st.evictions;
        }
        at[key] = slots.size();
        slots.push_back(key);
        ++st.misses;
      }
    }
  }
  *out = st;
  return K3MOE_OK;
}
