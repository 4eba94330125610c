"""The cache-policy simulator (host code of the C ABI; no GPU): LRU, Belady's MIN and random
replacement over traces of layer calls, each call a set of experts needed resident at once.

Pins: the textbook reference string whose page-fault counts under LRU and OPT are printed in
operating-systems texts; exhaustive search for the fewest misses on tiny batched traces (MIN
must reach it); a direct re-statement of the device cache's LRU rule (hits touched first, then
misses replace the least recently used slot); invariants that hold for every policy."""
import itertools
import random

import pytest

import mxfp4_routed_expert_06_b300 as k3

LRU, MIN, RND = k3.K3MOE_POLICY_LRU, k3.K3MOE_POLICY_MIN, k3.K3MOE_POLICY_RANDOM


def _singles(seq):
    return [[x] for x in seq]


def test_reference_string_fault_counts():
    # Silberschatz et al., Operating System Concepts, the 20-reference string with 3 frames:
    # OPT 9 page faults, LRU 12 page faults
    ref = [7, 0, 1, 2, 0, 3, 0, 4, 2, 3, 0, 3, 2, 1, 2, 0, 1, 7, 0, 1]
    assert k3.k3moe_cache_simulate(_singles(ref), 3, MIN)["misses"] == 9
    assert k3.k3moe_cache_simulate(_singles(ref), 3, LRU)["misses"] == 12


def _lru_direct(calls, n_slots):
    order = []  # front = most recent
    hits = misses = ev = 0
    for call in calls:
        miss = []
        for key in call:
            if key in order:
                order.remove(key)
                order.insert(0, key)
                hits += 1
            else:
                miss.append(key)
        for key in miss:
            if len(order) == n_slots:
                order.pop()
                ev += 1
            order.insert(0, key)
            misses += 1
    return {"hits": hits, "misses": misses, "evictions": ev}


def _fewest_misses(calls, n_slots):
    """Exhaustive search over every eviction choice (tiny traces only)."""
    best = [None]

    def rec(c, resident, misses):
        if best[0] is not None and misses >= best[0]:
            return
        if c == len(calls):
            best[0] = misses
            return
        need = calls[c]
        new = [x for x in need if x not in resident]
        keep = [x for x in resident if x in need]
        others = [x for x in resident if x not in need]
        room = n_slots - len(resident)
        n_evict = max(0, len(new) - room)
        for out in itertools.combinations(others, n_evict):
            nxt = frozenset(keep) | frozenset(x for x in others if x not in out) | frozenset(new)
            rec(c + 1, nxt, misses + len(new))

    rec(0, frozenset(), 0)
    return best[0]


def _random_trace(rng, n_calls, n_keys, max_call):
    return [rng.sample(range(n_keys), rng.randint(1, max_call)) for _ in range(n_calls)]


@pytest.mark.parametrize("seed", range(12))
def test_min_reaches_the_fewest_misses(seed):
    rng = random.Random(seed)
    n_slots = rng.randint(2, 4)
    calls = _random_trace(rng, rng.randint(4, 8), rng.randint(n_slots + 1, 7), min(2, n_slots))
    opt = _fewest_misses(calls, n_slots)
    got = k3.k3moe_cache_simulate(calls, n_slots, MIN)
    assert got["misses"] == opt
    assert k3.k3moe_cache_simulate(calls, n_slots, LRU)["misses"] >= opt
    assert k3.k3moe_cache_simulate(calls, n_slots, RND, seed)["misses"] >= opt


@pytest.mark.parametrize("seed", range(8))
def test_lru_follows_the_device_rule(seed):
    rng = random.Random(100 + seed)
    n_slots = rng.randint(3, 12)
    calls = _random_trace(rng, 200, 30, min(6, n_slots))
    assert k3.k3moe_cache_simulate(calls, n_slots, LRU) == _lru_direct(calls, n_slots)


@pytest.mark.parametrize("policy", [LRU, MIN, RND])
def test_invariants(policy):
    rng = random.Random(7)
    calls = _random_trace(rng, 300, 64, 16)
    total = sum(len(c) for c in calls)
    distinct = len({x for c in calls for x in c})
    for n_slots in (16, 40, 64, 100):
        st = k3.k3moe_cache_simulate(calls, n_slots, policy, 3)
        assert st["hits"] + st["misses"] == total
        assert st["evictions"] == max(0, st["misses"] - n_slots)  # empty slots fill first
        if n_slots >= distinct:  # everything fits: only cold misses
            assert st["misses"] == distinct and st["evictions"] == 0
    # random replacement is reproducible for one seed
    assert k3.k3moe_cache_simulate(calls, 20, RND, 11) == k3.k3moe_cache_simulate(calls, 20, RND, 11)


def test_min_is_never_worse():
    rng = random.Random(21)
    calls = _random_trace(rng, 400, 80, 8)
    for n_slots in (8, 16, 32, 60):
        m = k3.k3moe_cache_simulate(calls, n_slots, MIN)["misses"]
        assert m <= k3.k3moe_cache_simulate(calls, n_slots, LRU)["misses"]
        for s in range(3):
            assert m <= k3.k3moe_cache_simulate(calls, n_slots, RND, s)["misses"]


def test_refusals():
    with pytest.raises(k3.K3MoEError) as e:
        k3.k3moe_cache_simulate([[1, 2, 1]], 4, LRU)  # a key repeated within a call
    assert e.value.code == k3.K3MOE_ERR_INVALID_ARG
    with pytest.raises(k3.K3MoEError) as e:
        k3.k3moe_cache_simulate([[1, 2, 3]], 2, MIN)  # a call larger than the cache
    assert e.value.code == k3.K3MOE_ERR_BUDGET_TOO_SMALL
    with pytest.raises(k3.K3MoEError) as e:
        k3.k3moe_cache_simulate([[1]], 0, LRU)
    assert e.value.code == k3.K3MOE_ERR_INVALID_ARG
    with pytest.raises(k3.K3MoEError) as e:
        k3.k3moe_cache_simulate([[1]], 2, 9)
    assert e.value.code == k3.K3MOE_ERR_INVALID_ARG
    assert k3.k3moe_cache_simulate([], 2, LRU) == {"hits": 0, "misses": 0, "evictions": 0}
