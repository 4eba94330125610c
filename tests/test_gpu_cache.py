"""The device LRU expert cache ("four reductions", expert LRU paragraph): outputs do not depend
on the memory budget.

A cache-mode layer keeps its packed experts in a pinned host pool and copies the ones a call
needs into device slots.  Stacked layers (residual x_next = bf16_rne(y + x) between them, as a
caller would apply it) run under several budgets; every y must be byte-identical to the run
with the experts resident on the device, and the cache statistics must add up.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import GAP_MIN, assert_routing_matches, assert_routing_valid, assert_y_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import mxfp4_routed_expert_06_b300 as k3  # noqa: E402


EPS = 1e-6


def _run_stack(layers, x0, T, steps, d):
    """Run `steps` calls of T tokens through the stacked layers.  Layer 0 takes the token; after
    layer l the residual stream is r = bf16(r + y) and layer l+1 takes the RMSNorm of r (both
    from k3moe_residual_rmsnorm).  Returns the y of every (step, layer) as one uint8 array and
    the input of every layer call."""
    ys, xs = [], []
    for s in range(steps):
        r = x0[s].clone()
        x = x0[s]
        for L in layers:
            y = torch.empty((T, d), dtype=torch.float32, device="cuda")
            k3.k3moe_layer_forward(L, x, T, y)
            xs.append(x)
            ys.append(y)
            x = torch.empty_like(r)
            k3.k3moe_residual_rmsnorm(y, r, T, d, EPS, r, x)
    torch.cuda.synchronize()
    return torch.stack(ys).cpu().numpy().view(np.uint8), [a.cpu().numpy().view(np.uint16) for a in xs]


def test_residual_rmsnorm_matches_oracle():
    rng = np.random.default_rng(9)
    for T, d, scale in [(5, 7168, 2400.0), (3, 100, 1.0), (1, 1, 3.0), (2, 4096, 1e-3)]:
        x = synth.tokens_bf16(9, 0, 0, T, d)
        y = (rng.standard_normal((T, d)) * scale).astype(np.float32)
        xn_o, xr_o = oracle.residual_rmsnorm(y, x, EPS)
        xd = torch.from_numpy(x.view(np.int16)).cuda()
        yd = torch.from_numpy(y).cuda()
        nxt = torch.empty_like(xd)
        nrm = torch.empty_like(xd)
        k3.k3moe_residual_rmsnorm(yd, xd, T, d, EPS, nxt, nrm)
        k3.k3moe_residual_rmsnorm(yd, xd, T, d, EPS, xd, nrm)  # in place on the residual stream
        torch.cuda.synchronize()
        nxt_h = nxt.cpu().numpy().view(np.uint16)
        assert np.array_equal(nxt_h, xn_o), f"T={T} d={d}: residual differs"
        assert np.array_equal(xd.cpu().numpy().view(np.uint16), xn_o), "in-place residual differs"
        # the norm's sum of squares runs in another order and precision: one bf16 step at most,
        # where the fp64 value lies near a rounding boundary
        a = nrm.cpu().numpy().view(np.int16).astype(np.int32)
        b = xr_o.view(np.int16).astype(np.int32)
        assert np.abs(a - b).max() <= 1, f"T={T} d={d}: norm differs by more than one bf16 step"
        assert (a == b).mean() >= 0.99


def _distinct_per_call(layers, xs, T, k, n_layers):
    """Number of distinct experts each layer call routes to (from the library's own top-k)."""
    out = []
    for i, x in enumerate(xs):
        L = layers[i % n_layers]
        idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, k), dtype=torch.float32, device="cuda")
        xd = torch.from_numpy(x.view(np.int16)).cuda()
        k3.k3moe_router_topk(L, xd, T, idx, w)
        out.append((i % n_layers, np.unique(idx.cpu().numpy())))
    return out


def test_small_stack_budgets_bit_identical():
    d, f, E, k, T, n_layers, steps = 512, 256, 64, 6, 3, 2, 24
    dm = k3.dims(d, f, E, k, T)
    eb = k3.k3moe_packed_expert_bytes(dm)
    host = [synth.experts(5, l, 0, E, d, f) for l in range(n_layers)]
    Wr = [synth.router_weights(5, l, E, d) for l in range(n_layers)]
    x0 = [torch.from_numpy(synth.tokens_bf16(5, 0, s * T, T, d).view(np.int16)).cuda() for s in range(steps)]

    dev_layers = [k3.k3moe_pack_experts(dm, host[l][0], host[l][1], 0, Wr[l]) for l in range(n_layers)]
    y_ref, xs = _run_stack(dev_layers, x0, T, steps, d)
    used = _distinct_per_call(dev_layers, xs, T, k, n_layers)
    need = max(len(u) for _, u in used)
    total_distinct = len({(l, int(e)) for l, u in used for e in u})

    # oracle on the first step of every layer (per-layer parity on the GPU chain's inputs)
    for l in range(n_layers):
        x = xs[l]
        ref = oracle.layer(x, Wr[l], None, k, f, host[l][0], host[l][1])
        ok = oracle.topk_gap(ref["keys"], k) >= GAP_MIN
        assert ok.sum() >= 2
        y = y_ref.view(np.float32).reshape(steps * n_layers, T, d)[l]
        idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, k), dtype=torch.float32, device="cuda")
        k3.k3moe_router_topk(dev_layers[l], torch.from_numpy(x.view(np.int16)).cuda(), T, idx, w)
        assert_routing_matches(idx.cpu().numpy()[ok], w.cpu().numpy()[ok], ref["idx"][ok], ref["w"][ok],
                               ref["keys"][ok])
        assert_y_close(y[ok], ref["y"][ok], ref["sumabs"][ok], f"layer {l}")

    cache_layers, caches = None, []
    for slots in (need, need + 7, 2 * E):
        caches.append(k3.k3moe_cache_create(slots * eb, eb))
        cache = caches[-1]
        if cache_layers is None:
            cache_layers = [k3.k3moe_pack_experts(dm, host[l][0], host[l][1], 0, Wr[l], None, cache)
                            for l in range(n_layers)]
        else:
            for L in cache_layers:
                k3.k3moe_layer_set_cache(L, cache)
        y, _ = _run_stack(cache_layers, x0, T, steps, d)
        assert np.array_equal(y, y_ref), f"{slots} slots: output differs from the device-resident run"
        st = k3.k3moe_cache_stats(cache)
        assert st["calls"] == steps * n_layers
        assert st["hits"] + st["misses"] == sum(len(u) for _, u in used)
        # the host simulator's LRU replays the same trace to the same counts
        trace = [[l * E + int(e) for e in u] for l, u in used]
        sim = k3.k3moe_cache_simulate(trace, slots, k3.K3MOE_POLICY_LRU)
        assert (st["hits"], st["misses"], st["evictions"]) == (sim["hits"], sim["misses"], sim["evictions"])
        assert st["h2d_bytes"] == st["misses"] * eb
        if slots >= n_layers * E:
            assert st["evictions"] == 0 and st["misses"] == total_distinct
        else:
            assert st["misses"] > total_distinct  # something was evicted and brought back
        # a second pass with the cache warm: only which copies run may change
        k3.k3moe_cache_reset_stats(cache)
        y2, _ = _run_stack(cache_layers, x0, T, steps, d)
        assert np.array_equal(y2, y_ref)
        st2 = k3.k3moe_cache_stats(cache)
        if slots >= n_layers * E:
            assert st2["misses"] == 0 and st2["hits"] == st["hits"] + st["misses"]
        sim2 = k3.k3moe_cache_simulate(trace + trace, slots, k3.K3MOE_POLICY_LRU)
        assert [st2[n] for n in ("hits", "misses", "evictions")] == [sim2[n] - sim[n] for n in
                                                                     ("hits", "misses", "evictions")]
    for L in cache_layers + dev_layers:
        k3.k3moe_layer_free(L)
    for c in caches:
        k3.k3moe_cache_destroy(c)


@pytest.mark.parametrize("fail_at,slots,miss_path", [(1, 64, 0), (3, 64, 0), (6, 10, 0), (1, 64, 1), (6, 10, 1)])
def test_failed_expert_copy_reports_error_then_recovers(fail_at, slots, miss_path):
    """A cache-miss copy that fails (injected on the host: the copy call reports an error and
    copies nothing) makes that forward return K3MOE_ERR_CUDA; the slot it was filling is
    forgotten, so the following calls copy the expert again and give the device-resident
    output, byte for byte.  miss_path 1: the zero-copy miss path (the misses listed before the
    failing one are still copied by the kernel)."""
    d, f, E, k, T, steps = 512, 256, 32, 4, 2, 6
    dm = k3.dims(d, f, E, k, T)
    eb = k3.k3moe_packed_expert_bytes(dm)
    nib, scl = synth.experts(9, 0, 0, E, d, f)
    Wr = synth.router_weights(9, 0, E, d)
    xs = [torch.from_numpy(synth.tokens_bf16(9, 0, s * T, T, d).view(np.int16)).cuda() for s in range(steps)]
    ref_layer = k3.k3moe_pack_experts(dm, nib, scl, 0, Wr)
    cache = k3.k3moe_cache_create(slots * eb, eb)
    layer = k3.k3moe_pack_experts(dm, nib, scl, 0, Wr, None, cache)
    k3.k3moe_set_option(layer, k3.K3MOE_OPT_MISS_PATH, miss_path)
    try:
        refs = []
        for x in xs:
            y = torch.empty((T, d), dtype=torch.float32, device="cuda")
            k3.k3moe_layer_forward(ref_layer, x, T, y)
            refs.append(y)
        torch.cuda.synchronize()
        k3.k3moe_set_option(layer, k3.K3MOE_OPT_TEST_FAIL_COPY, fail_at)
        y = torch.empty((T, d), dtype=torch.float32, device="cuda")
        with pytest.raises(k3.K3MoEError) as ei:
            for x in xs:  # the failure comes on the fail_at-th miss, in whichever call makes it
                k3.k3moe_layer_forward(layer, x, T, y)
                torch.cuda.synchronize()
        assert ei.value.code == k3.K3MOE_ERR_CUDA and "cache slot" in str(ei.value)
        for _ in range(2):  # every later call is whole again, cold slots or warm
            for x, r in zip(xs, refs):
                y = torch.empty((T, d), dtype=torch.float32, device="cuda")
                k3.k3moe_layer_forward(layer, x, T, y)
                torch.cuda.synchronize()
                assert torch.equal(y, r)
        st = k3.k3moe_cache_stats(cache)
        assert st["h2d_bytes"] == st["misses"] * eb
    finally:
        k3.k3moe_layer_free(layer)
        k3.k3moe_layer_free(ref_layer)
        k3.k3moe_cache_destroy(cache)


def test_zero_copy_miss_path_matches_copy_engine():
    """Two stacked layers sharing a cache that holds about half their experts: the zero-copy miss
    path (one kernel per call reads the misses from the mapped pinned pool) gives the same bytes
    as the device-resident layers, and the same hits, misses and evictions as the copy-engine
    path (the bookkeeping is shared; only how the bytes travel differs)."""
    d, f, E, k, T, n_layers, steps = 512, 256, 32, 4, 3, 2, 16
    dm = k3.dims(d, f, E, k, T)
    eb = k3.k3moe_packed_expert_bytes(dm)
    host = [synth.experts(15, l, 0, E, d, f) for l in range(n_layers)]
    Wr = [synth.router_weights(15, l, E, d) for l in range(n_layers)]
    x0 = [torch.from_numpy(synth.tokens_bf16(15, 0, s * T, T, d).view(np.int16)).cuda() for s in range(steps)]
    dev = [k3.k3moe_pack_experts(dm, host[l][0], host[l][1], 0, Wr[l]) for l in range(n_layers)]
    y_ref, _ = _run_stack(dev, x0, T, steps, d)
    stats = {}
    for miss_path in (k3.K3MOE_MISS_COPY_ENGINE, k3.K3MOE_MISS_ZERO_COPY):
        cache = k3.k3moe_cache_create(E * eb, eb)
        layers = [k3.k3moe_pack_experts(dm, host[l][0], host[l][1], 0, Wr[l], None, cache) for l in range(n_layers)]
        for L in layers:
            k3.k3moe_set_option(L, k3.K3MOE_OPT_MISS_PATH, miss_path)
        y, _ = _run_stack(layers, x0, T, steps, d)
        assert np.array_equal(y, y_ref), f"miss path {miss_path}: y differs from the device-resident layers"
        st = k3.k3moe_cache_stats(cache)
        assert st["misses"] > 0 and st["evictions"] > 0 and st["h2d_bytes"] == st["misses"] * eb
        stats[miss_path] = (st["hits"], st["misses"], st["evictions"])
        for L in layers:
            k3.k3moe_layer_free(L)
        k3.k3moe_cache_destroy(cache)
    assert stats[k3.K3MOE_MISS_COPY_ENGINE] == stats[k3.K3MOE_MISS_ZERO_COPY]
    for L in dev:
        k3.k3moe_layer_free(L)


def test_device_side_lru_matches_host_bookkeeping():
    """The cache with its LRU state on the device (lookup kernel + zero-copy miss copies, no host
    round trip): the same bytes as the device-resident layers and the same hits, misses and
    evictions as the host bookkeeping, also across a move to another device-side cache; layers
    that might need more experts than the cache has slots are refused when they attach."""
    d, f, E, k, T, n_layers, steps = 512, 256, 32, 4, 3, 2, 16
    dm = k3.dims(d, f, E, k, T)
    eb = k3.k3moe_packed_expert_bytes(dm)
    host = [synth.experts(17, l, 0, E, d, f) for l in range(n_layers)]
    Wr = [synth.router_weights(17, l, E, d) for l in range(n_layers)]
    x0 = [torch.from_numpy(synth.tokens_bf16(17, 0, s * T, T, d).view(np.int16)).cuda() for s in range(steps)]
    dev = [k3.k3moe_pack_experts(dm, host[l][0], host[l][1], 0, Wr[l]) for l in range(n_layers)]
    y_ref, _ = _run_stack(dev, x0, T, steps, d)
    stats = {}
    for device_lru in (0, 1):
        cache = k3.k3moe_cache_create(E * eb, eb)
        k3.k3moe_cache_set_device_lru(cache, device_lru)
        layers = [k3.k3moe_pack_experts(dm, host[l][0], host[l][1], 0, Wr[l], None, cache) for l in range(n_layers)]
        if device_lru:
            with pytest.raises(k3.K3MoEError) as ei:  # layers attached: the mode is fixed
                k3.k3moe_cache_set_device_lru(cache, 0)
            assert ei.value.code == k3.K3MOE_ERR_INVALID_ARG
        y, _ = _run_stack(layers, x0, T, steps, d)
        assert np.array_equal(y, y_ref), f"device_lru={device_lru}: y differs from the device-resident layers"
        st = k3.k3moe_cache_stats(cache)
        assert st["misses"] > 0 and st["evictions"] > 0 and st["h2d_bytes"] == st["misses"] * eb
        stats[device_lru] = (st["hits"], st["misses"], st["evictions"], st["calls"])
        if device_lru:
            other = k3.k3moe_cache_create(E * eb, eb)
            k3.k3moe_cache_set_device_lru(other, 1)
            for L in layers:
                k3.k3moe_layer_set_cache(L, other)
            y2, _ = _run_stack(layers, x0, T, steps, d)
            assert np.array_equal(y2, y_ref)
            st2 = k3.k3moe_cache_stats(other)
            assert st2["misses"] > 0 and st2["calls"] == steps * n_layers
        for L in layers:
            k3.k3moe_layer_free(L)
        k3.k3moe_cache_destroy(cache)
        if device_lru:
            k3.k3moe_cache_destroy(other)
    assert stats[0] == stats[1]
    tiny = k3.k3moe_cache_create(10 * eb, eb)  # T_max * k = 12 experts may be needed at once
    k3.k3moe_cache_set_device_lru(tiny, 1)
    with pytest.raises(k3.K3MoEError) as ei:
        k3.k3moe_pack_experts(dm, host[0][0], host[0][1], 0, Wr[0], None, tiny)
    assert ei.value.code == k3.K3MOE_ERR_BUDGET_TOO_SMALL
    k3.k3moe_cache_destroy(tiny)
    for L in dev:
        k3.k3moe_layer_free(L)


def test_budget_too_small_then_recovers():
    d, f, E, k, T = 256, 128, 16, 4, 2
    dm = k3.dims(d, f, E, k, T)
    eb = k3.k3moe_packed_expert_bytes(dm)
    nib, scl = synth.experts(8, 0, 0, E, d, f)
    Wr = synth.router_weights(8, 0, E, d)
    x = torch.from_numpy(synth.tokens_bf16(8, 0, 0, T, d).view(np.int16)).cuda()
    small = k3.k3moe_cache_create(3 * eb, eb)  # a call needs at least k = 4 experts
    L = k3.k3moe_pack_experts(dm, nib, scl, 0, Wr, None, small)
    y = torch.empty((T, d), dtype=torch.float32, device="cuda")
    with pytest.raises(k3.K3MoEError) as ei:
        k3.k3moe_layer_forward(L, x, T, y)
    assert ei.value.code == k3.K3MOE_ERR_BUDGET_TOO_SMALL
    big = k3.k3moe_cache_create(E * eb, eb)
    k3.k3moe_layer_set_cache(L, big)
    k3.k3moe_layer_forward(L, x, T, y)
    D = k3.k3moe_pack_experts(dm, nib, scl, 0, Wr)
    y_ref = torch.empty_like(y)
    k3.k3moe_layer_forward(D, x, T, y_ref)
    torch.cuda.synchronize()
    assert torch.equal(y, y_ref)
    with pytest.raises(k3.K3MoEError):
        k3.k3moe_layer_set_cache(D, big)  # packed without a cache
    k3.k3moe_layer_free(L)
    k3.k3moe_layer_free(D)
    k3.k3moe_cache_destroy(small)
    k3.k3moe_cache_destroy(big)


K3 = dict(d=7168, f=1536, E=896, k=16)
GB = 1_000_000_000


def _free_host_gb():
    try:
        with open("/proc/meminfo") as fh:
            for ln in fh:
                if ln.startswith("MemAvailable:"):
                    return int(ln.split()[1]) * 1024 / GB
    except OSError:
        pass
    return 0.0


def test_k3_four_layers_budgets_bit_identical():
    """Four stacked K3 layers (62.9 GB pinned pool), T=1 decode for 256 steps, budgets of 8,
    24 and 64 GB: the y of every step and layer is byte-identical across budgets; the routing of
    all 1024 layer calls matches the oracle on the chain's own inputs (exact where the 16th/17th
    keys are separated, a valid top-k within fp32 rounding elsewhere); y of steps 0-15 of every
    layer matches the oracle."""
    d, f, E, k = K3["d"], K3["f"], K3["E"], K3["k"]
    n_layers, steps, T = 4, 256, 1
    eb = k3.k3moe_packed_expert_bytes(k3.dims(d, f, E, k, T))
    if _free_host_gb() < n_layers * E * eb / GB + 20:
        pytest.skip("not enough host memory for the 4-layer pinned pool")
    nb, sb = synth.expert_bytes(d, f)
    cache = k3.k3moe_cache_create(8 * GB, eb)
    layers, Wr = [], []
    for l in range(n_layers):
        dn = torch.empty(E * nb, dtype=torch.uint8, device="cuda")
        ds = torch.empty(E * sb, dtype=torch.uint8, device="cuda")
        synth.experts_to_device(11, l, 0, E, d, f, dn.data_ptr(), ds.data_ptr())
        Wr.append(synth.router_weights(11, l, E, d))
        layers.append(k3.k3moe_pack_experts(k3.dims(d, f, E, k, T), dn, ds, 1, torch.from_numpy(Wr[l]).cuda(),
                                            None, cache))
        del dn, ds
        torch.cuda.synchronize()
        torch.cuda.empty_cache()

    # step s takes token s; the oracle comparison below skips layer calls whose input lies
    # within GAP_MIN of a top-k tie (the byte comparison across budgets needs no such filter)
    x0 = []
    for s in range(steps):
        x0.append(torch.from_numpy(synth.tokens_bf16(11, 0, s, 1, d).view(np.int16)).cuda())

    results, stats, caches = {}, {}, [cache]
    for budget in (8, 24, 64):
        if budget != 8:
            caches.append(k3.k3moe_cache_create(budget * GB, eb))
            for L in layers:
                k3.k3moe_layer_set_cache(L, caches[-1])
        y, xs = _run_stack(layers, x0, T, steps, d)
        results[budget] = y
        stats[budget] = k3.k3moe_cache_stats(caches[-1])
    assert np.array_equal(results[8], results[24]) and np.array_equal(results[8], results[64])
    for budget, st in stats.items():
        assert st["calls"] == steps * n_layers
        assert st["hits"] + st["misses"] == steps * n_layers * k  # T=1: k distinct experts per call
        assert st["h2d_bytes"] == st["misses"] * eb
    assert stats[64]["evictions"] == 0
    assert stats[8]["misses"] > stats[24]["misses"] > stats[64]["misses"]

    # oracle routing of every layer call, on the chain's own inputs
    for l in range(n_layers):
        xl = np.concatenate(xs[l::n_layers])
        xd = torch.from_numpy(xl.view(np.int16)).cuda()
        idx = torch.empty((steps, k), dtype=torch.int32, device="cuda")
        w = torch.empty((steps, k), dtype=torch.float32, device="cuda")
        for s in range(steps):  # T=1 calls, as the layers ran them
            k3.k3moe_router_topk(layers[l], xd[s:s + 1], 1, idx[s:s + 1], w[s:s + 1])
        torch.cuda.synchronize()
        idx_h, w_h = idx.cpu().numpy(), w.cpu().numpy()
        i_o, w_o, lg_o, keys = oracle.router(xl, Wr[l], None, k)
        sep = oracle.topk_gap(keys, k) >= GAP_MIN
        assert_routing_matches(idx_h[sep], w_h[sep], i_o[sep], w_o[sep], keys[sep])
        assert_routing_valid(idx_h[~sep], w_h[~sep], lg_o[~sep], keys[~sep], 1e-5)

    # oracle y: steps 0-15 of every layer, on the chain's own inputs
    yv = results[8].view(np.float32).reshape(steps * n_layers, d)
    checked = 0
    for i in range(16 * n_layers):
        l = i % n_layers
        x = xs[i]
        idx_o, w_o, _, keys = oracle.router(x, Wr[l], None, k)
        if oracle.topk_gap(keys, k)[0] < GAP_MIN:
            continue
        flat = idx_o.reshape(-1)
        nibs, scls = [], []
        for e in flat:
            n_, s_ = synth.experts(11, l, int(e), int(e) + 1, d, f)
            nibs.append(n_[0])
            scls.append(s_[0])
        y_o, sumabs = oracle.moe(x, w_o, nibs, scls, f)
        assert_y_close(yv[i:i + 1], y_o, sumabs, f"step {i // n_layers} layer {l}")
        checked += 1
    assert checked >= 32  # about 30% of random tokens have their 16th/17th keys within 1e-3
    for L in layers:
        k3.k3moe_layer_free(L)
    for c in caches:
        k3.k3moe_cache_destroy(c)
