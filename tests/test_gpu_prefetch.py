"""Expert prefetch into the cache ("four reductions", expert LRU paragraph: the engine's cache
loads the experts of a batch ahead of the arithmetic).

k3moe_cache_prefetch copies listed experts of a cache-mode layer into slots on the cache's copy
stream before the call that needs them.  Checked here:
  * a prefetched expert is a hit for the next call, and the output is the device-resident
    layer's, byte for byte;
  * a prefetch never takes a slot that a call still in flight may read, nor one holding an
    expert it lists: the number it copies is exactly the number of slots it may take;
  * after k3moe_sync every slot may be taken again;
  * stacked layers with the next call's experts prefetched (exact, or wrong guesses) give the
    bytes of the run without prefetch;
  * an injected copy failure is reported and forgotten; the refusals.
"""
import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import mxfp4_routed_expert_06_b300 as k3  # noqa: E402

EPS = 1e-6
d, f, E, k = 512, 256, 32, 4


def _tok(seed, i, T=1):
    return torch.from_numpy(synth.tokens_bf16(seed, 0, i * T, T, d).view(np.int16)).cuda()


def _experts_of(layer, x, T=1):
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    k3.k3moe_router_topk(layer, x, T, idx, w)
    return np.unique(idx.cpu().numpy()).astype(np.int32)


def _forward(layer, x, T=1):
    y = torch.empty((T, d), dtype=torch.float32, device="cuda")
    k3.k3moe_layer_forward(layer, x, T, y)
    return y


def _layers(seed, slots, T=1):
    dm = k3.dims(d, f, E, k, T)
    eb = k3.k3moe_packed_expert_bytes(dm)
    nib, scl = synth.experts(seed, 0, 0, E, d, f)
    Wr = synth.router_weights(seed, 0, E, d)
    ref = k3.k3moe_pack_experts(dm, nib, scl, 0, Wr)
    cache = k3.k3moe_cache_create(slots * eb, eb)
    layer = k3.k3moe_pack_experts(dm, nib, scl, 0, Wr, None, cache)
    return ref, cache, layer, eb


def test_prefetch_hits_and_never_takes_a_slot_in_flight():
    ref, cache, layer, eb = _layers(21, 16)
    try:
        xa, xb = _tok(21, 0), _tok(21, 1)
        sa, sb = _experts_of(ref, xa), _experts_of(ref, xb)
        ya_ref, yb_ref = _forward(ref, xa), _forward(ref, xb)
        torch.cuda.synchronize()

        # a cold cache: the prefetch copies all of a's experts, and a's call then only hits
        assert k3.k3moe_cache_prefetch(layer, sa) == len(sa)
        ya = _forward(layer, xa)
        torch.cuda.synchronize()
        st = k3.k3moe_cache_stats(cache)
        assert (st["prefetched"], st["hits"], st["misses"]) == (len(sa), len(sa), 0)
        assert torch.equal(ya, ya_ref)

        # b's call is queued and not waited for: its slots are in flight.  A prefetch of 16
        # experts outside b's set may take only the 16 - |b| other slots, less those holding
        # listed experts (they are kept and become most recently used).
        yb = _forward(layer, xb)
        others = np.array([e for e in range(E) if e not in set(sb.tolist())][:16], np.int32)
        resident_listed = len(set(others.tolist()) & (set(sa.tolist()) - set(sb.tolist())))
        got = k3.k3moe_cache_prefetch(layer, others)
        assert got == 16 - len(sb) - resident_listed
        torch.cuda.synchronize()
        assert torch.equal(yb, yb_ref)

        # b's experts are still resident: the same call again only hits
        k3.k3moe_sync(layer)
        k3.k3moe_cache_reset_stats(cache)
        yb2 = _forward(layer, xb)
        torch.cuda.synchronize()
        st = k3.k3moe_cache_stats(cache)
        assert (st["hits"], st["misses"]) == (len(sb), 0)
        assert torch.equal(yb2, yb_ref)

        # a prefetch never evicts an expert it lists: listing every expert copies none
        k3.k3moe_sync(layer)
        assert k3.k3moe_cache_prefetch(layer, np.arange(E, dtype=np.int32)) == 0

        # after k3moe_sync any slot may be taken: 8 experts that are not resident all come in
        k3.k3moe_sync(layer)
        k3.k3moe_cache_reset_stats(cache)
        absent = [e for e in range(E) if e not in set(others.tolist()) | set(sb.tolist())
                  | set(sa.tolist())][:8]
        assert len(absent) == 8
        assert k3.k3moe_cache_prefetch(layer, absent + absent) == 8  # duplicates are no-ops
        st = k3.k3moe_cache_stats(cache)
        assert st["prefetched"] == 8 and st["evictions"] == 8 and st["h2d_bytes"] == 8 * eb
        for x, y_ref in ((xa, ya_ref), (xb, yb_ref)):  # whatever was evicted, outputs are whole
            y = _forward(layer, x)
            torch.cuda.synchronize()
            assert torch.equal(y, y_ref)
    finally:
        k3.k3moe_layer_free(layer)
        k3.k3moe_layer_free(ref)
        k3.k3moe_cache_destroy(cache)


def _stack(layers, x0, hook=None):
    """T=1 tokens through stacked layers (r = bf16(r + y), next layer takes RMSNorm(r)).
    hook(call_index) runs right after each layer call is queued."""
    ys, c = [], 0
    for x in x0:
        r = x.clone()
        for L in layers:
            y = _forward(L, x)
            if hook:
                hook(c)
            c += 1
            ys.append(y)
            x = torch.empty_like(r)
            k3.k3moe_residual_rmsnorm(y, r, 1, d, EPS, r, x)
    torch.cuda.synchronize()
    return torch.stack(ys).cpu().numpy().view(np.uint8)


def test_stacked_layers_with_prefetch_are_byte_identical():
    n_layers, steps, slots = 2, 12, 14
    dm = k3.dims(d, f, E, k, 1)
    eb = k3.k3moe_packed_expert_bytes(dm)
    host = [synth.experts(23, l, 0, E, d, f) for l in range(n_layers)]
    Wr = [synth.router_weights(23, l, E, d) for l in range(n_layers)]
    x0 = [_tok(23, s) for s in range(steps)]
    dev = [k3.k3moe_pack_experts(dm, host[l][0], host[l][1], 0, Wr[l]) for l in range(n_layers)]
    # each call's experts, from the device-resident run (the inputs of every call are the same)
    sets = []
    for x in x0:
        r = x.clone()
        for L in dev:
            sets.append(_experts_of(L, x))
            y = _forward(L, x)
            x = torch.empty_like(r)
            k3.k3moe_residual_rmsnorm(y, r, 1, d, EPS, r, x)
    y_ref = _stack(dev, x0)
    rng = np.random.default_rng(23)
    results = {}
    try:
        for mode in ("none", "exact", "wrong"):
            cache = k3.k3moe_cache_create(slots * eb, eb)
            layers = [k3.k3moe_pack_experts(dm, host[l][0], host[l][1], 0, Wr[l], None, cache)
                      for l in range(n_layers)]
            n_calls = steps * n_layers

            def hook(c):
                if mode == "none" or c + 1 == n_calls:
                    return
                nxt = layers[(c + 1) % n_layers]
                ids = sets[c + 1] if mode == "exact" else rng.choice(E, size=6, replace=False)
                k3.k3moe_cache_prefetch(nxt, ids)

            if mode != "none":
                k3.k3moe_cache_prefetch(layers[0], sets[0] if mode == "exact" else [0, 1])
            y = _stack(layers, x0, hook)
            assert np.array_equal(y, y_ref), f"prefetch {mode}: y differs from the device-resident layers"
            st = k3.k3moe_cache_stats(cache)
            results[mode] = st
            assert st["h2d_bytes"] == (st["misses"] + st["prefetched"]) * eb
            assert st["calls"] == n_calls
            for L in layers:
                k3.k3moe_layer_free(L)
            k3.k3moe_cache_destroy(cache)
        # an exact prefetch leaves the calls nothing to copy: every expert is a hit
        assert results["exact"]["misses"] == 0
        assert results["exact"]["hits"] == sum(len(s) for s in sets)
        assert results["none"]["prefetched"] == 0 and results["wrong"]["prefetched"] > 0
    finally:
        for L in dev:
            k3.k3moe_layer_free(L)


def test_prefetch_copy_failure_is_forgotten_and_refusals():
    ref, cache, layer, eb = _layers(25, 16)
    try:
        xs = [_tok(25, i) for i in range(6)]
        refs = [_forward(ref, x) for x in xs]
        torch.cuda.synchronize()
        k3.k3moe_set_option(layer, k3.K3MOE_OPT_TEST_FAIL_COPY, 2)
        with pytest.raises(k3.K3MoEError) as ei:
            k3.k3moe_cache_prefetch(layer, [3, 7, 11, 19])
        assert ei.value.code == k3.K3MOE_ERR_CUDA and "prefetching expert 7" in str(ei.value)
        for _ in range(2):
            for x, r in zip(xs, refs):
                y = _forward(layer, x)
                torch.cuda.synchronize()
                assert torch.equal(y, r)
        st = k3.k3moe_cache_stats(cache)
        assert st["prefetched"] == 1 and st["h2d_bytes"] == (st["misses"] + 1) * eb

        for bad in ([E], [-1], [0, 5, E + 3]):
            with pytest.raises(k3.K3MoEError) as ei:
                k3.k3moe_cache_prefetch(layer, bad)
            assert ei.value.code == k3.K3MOE_ERR_INVALID_ARG
        assert k3.k3moe_cache_prefetch(layer, []) == 0
        with pytest.raises(k3.K3MoEError) as ei:  # experts resident on the device: no cache
            k3.k3moe_cache_prefetch(ref, [0])
        assert ei.value.code == k3.K3MOE_ERR_INVALID_ARG
        dl = k3.k3moe_cache_create(16 * eb, eb)
        k3.k3moe_cache_set_device_lru(dl, 1)
        k3.k3moe_layer_set_cache(layer, dl)
        with pytest.raises(k3.K3MoEError) as ei:
            k3.k3moe_cache_prefetch(layer, [0])
        assert ei.value.code == k3.K3MOE_ERR_UNSUPPORTED
        k3.k3moe_layer_set_cache(layer, cache)
    finally:
        k3.k3moe_layer_free(layer)
        k3.k3moe_layer_free(ref)
        k3.k3moe_cache_destroy(cache)
        if "dl" in locals():
            k3.k3moe_cache_destroy(dl)
