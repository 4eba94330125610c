"""Parity of the tcgen05 grouped-GEMM path (large T) against the fp64 CPU oracle.

The path is forced with K3MOE_OPT_PATH = K3MOE_PATH_GEMM.  Routing and bucketing are the same
kernels as the register-decode path; y must be within 2e-3 * sum|terms| + 1e-5 per element.
Shapes cover ragged M-tiles (experts with a count that is not a multiple of 128), both N-tile
widths of the down projection (d % 256 == 0 and d % 256 == 128), K stage counts that are not a
multiple of the decoders' prefetch depth, scale spans up to the 36 steps the fp16 image holds
exactly (subnormal fp16 weights included), and the K3 shape with hot experts.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import assert_routing_matches, assert_y_close, gap_filtered_tokens

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import mxfp4_routed_expert_06_b300 as k3  # noqa: E402


def _dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def _forward(L, x, d, path):
    k3.k3moe_set_option(L, k3.K3MOE_OPT_PATH, path)
    T = x.shape[0]
    y = torch.empty((T, d), dtype=torch.float32, device="cuda")
    k3.k3moe_layer_forward(L, _dev(x), T, y)
    k3.k3moe_sync(L)
    return y.cpu().numpy()


@pytest.mark.parametrize("d,f,E,k,T,lo,hi", [
    (512, 256, 16, 4, 600, 121, 125),    # 2 M-tiles per expert (ragged), DN N-tile 256
    (384, 128, 8, 2, 300, 121, 125),     # d % 256 = 128: DN N-tile 128; 6 K stages
    (256, 128, 8, 2, 4, 121, 125),       # tiny: every tile mostly padding
    (1024, 384, 12, 3, 130, 121, 125),   # 3 gate/up N-tiles
    (512, 256, 16, 4, 200, 100, 136),    # span 36: smallest weights are fp16 subnormals
    (256, 128, 8, 2, 64, 0, 30),         # zero scale bytes (2^-127)
])
def test_gemm_path_matches_oracle(d, f, E, k, T, lo, hi):
    seed = 31
    nib, scl = synth.experts(seed, 0, 0, E, d, f, lo, hi)
    Wr = synth.router_weights(seed, 0, E, d)
    L = k3.k3moe_pack_experts(k3.dims(d, f, E, k, T), nib, scl, 0, Wr)
    x, _ = gap_filtered_tokens(seed, 0, 0, T, d, Wr, None, k)
    ref = oracle.layer(x, Wr, None, k, f, nib, scl)
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    k3.k3moe_router_topk(L, _dev(x), T, idx, w)
    torch.cuda.synchronize()
    assert_routing_matches(idx.cpu().numpy(), w.cpu().numpy(), ref["idx"], ref["w"], ref["keys"])
    y = _forward(L, x, d, k3.K3MOE_PATH_GEMM)
    assert_y_close(y, ref["y"], ref["sumabs"], f"gemm path d={d} f={f} E={E} k={k} T={T}")
    # deterministic: a second call is bitwise identical
    y2 = _forward(L, x, d, k3.K3MOE_PATH_GEMM)
    assert np.array_equal(y, y2)
    k3.k3moe_layer_free(L)


def test_gemm_refuses_too_wide_scale_span_and_auto_falls_back():
    d, f, E, k, T = 256, 128, 8, 2, 40
    nib, scl = synth.experts(3, 0, 0, E, d, f, 100, 140)  # span 40 > 36
    Wr = synth.router_weights(3, 0, E, d)
    L = k3.k3moe_pack_experts(k3.dims(d, f, E, k, T), nib, scl, 0, Wr)
    x, _ = gap_filtered_tokens(3, 0, 0, T, d, Wr, None, k)
    with pytest.raises(k3.K3MoEError) as ei:
        _forward(L, x, d, k3.K3MOE_PATH_GEMM)
    assert ei.value.code == k3.K3MOE_ERR_UNSUPPORTED
    k3.k3moe_set_option(L, k3.K3MOE_OPT_GEMM_MIN_T, 1)
    y = _forward(L, x, d, k3.K3MOE_PATH_AUTO)  # AUTO keeps the register-decode path
    ref = oracle.layer(x, Wr, None, k, f, nib, scl)
    assert_y_close(y, ref["y"], ref["sumabs"], "auto fallback")
    k3.k3moe_layer_free(L)


def test_gemm_path_k3_hot_experts():
    """K3 shape, T=256 with +2.0 bias on 32 experts (every token's top-16 lies among them):
    128 picks per hot expert on average.  Both FFN paths are checked element by element against
    the oracle on a seeded sample of tokens (plus the first and the last)."""
    d, f, E, k, T = 7168, 1536, 896, 16, 256
    nb, sb = synth.expert_bytes(d, f)
    dn = torch.empty(E * nb, dtype=torch.uint8, device="cuda")
    ds = torch.empty(E * sb, dtype=torch.uint8, device="cuda")
    synth.experts_to_device(41, 0, 0, E, d, f, dn.data_ptr(), ds.data_ptr())
    Wr = synth.router_weights(41, 0, E, d)
    bias = synth.hot_bias(41, 0, E, 32, 2.0)
    L = k3.k3moe_pack_experts(k3.dims(d, f, E, k, T), dn, ds, 1, _dev(Wr), _dev(bias))
    del dn, ds
    torch.cuda.empty_cache()
    x, _ = gap_filtered_tokens(41, 0, 0, T, d, Wr, bias, k)
    y_g = _forward(L, x, d, k3.K3MOE_PATH_GEMM)
    y_d = _forward(L, x, d, k3.K3MOE_PATH_DECODE)
    rng = np.random.default_rng(41)
    sample = sorted(set(rng.choice(np.arange(1, T - 1), size=14, replace=False).tolist()) | {0, T - 1})
    idx_o, w_o, _, keys = oracle.router(x[sample], Wr, bias, k)
    assert set(np.unique(idx_o).tolist()) <= set(np.nonzero(bias)[0].tolist())
    cache = {}
    nibs, scls = [], []
    for e in idx_o.reshape(-1).tolist():
        if e not in cache:
            n_, s_ = synth.experts(41, 0, e, e + 1, d, f)
            cache[e] = (n_[0], s_[0])
        nibs.append(cache[e][0])
        scls.append(cache[e][1])
    y_o, sumabs = oracle.moe(x[sample], w_o, nibs, scls, f)
    assert_y_close(y_g[sample], y_o, sumabs, "K3 T=256, tensor-core path")
    assert_y_close(y_d[sample], y_o, sumabs, "K3 T=256, register-decode path")
    k3.k3moe_layer_free(L)


def test_gemm_path_in_cache_mode_matches_device_resident():
    """Cache mode on the tensor-core path: two layers share a cache with fewer slots than their
    experts, so calls evict and copy; every y is byte-identical to the device-resident layers'."""
    d, f, E, k, T = 512, 256, 16, 4, 300
    dm = k3.dims(d, f, E, k, T)
    eb = k3.k3moe_packed_expert_bytes(dm)
    host = [synth.experts(57, l, 0, E, d, f) for l in range(2)]
    Wr = [synth.router_weights(57, l, E, d) for l in range(2)]
    dev = [k3.k3moe_pack_experts(dm, host[l][0], host[l][1], 0, Wr[l]) for l in range(2)]
    cache = k3.k3moe_cache_create((E + 5) * eb, eb)
    cached = [k3.k3moe_pack_experts(dm, host[l][0], host[l][1], 0, Wr[l], None, cache) for l in range(2)]
    try:
        for L in dev + cached:
            k3.k3moe_set_option(L, k3.K3MOE_OPT_PATH, k3.K3MOE_PATH_GEMM)
        order = [0, 1, 0, 1, 1, 0]
        for step, l in enumerate(order):
            x, _ = gap_filtered_tokens(57, l, step * T, T, d, Wr[l], None, k)
            y_ref = _forward(dev[l], x, d, k3.K3MOE_PATH_GEMM)
            y_c = _forward(cached[l], x, d, k3.K3MOE_PATH_GEMM)
            assert np.array_equal(y_ref.view(np.uint32), y_c.view(np.uint32)), f"step {step} layer {l}"
        st = k3.k3moe_cache_stats(cache)
        assert st["evictions"] > 0 and st["misses"] > E
        assert st["calls"] == len(order)
        # the last call's output against the oracle as well
        ref = oracle.layer(x, Wr[l], None, k, f, host[l][0], host[l][1])
        assert_y_close(y_c, ref["y"], ref["sumabs"], "cache-mode gemm path")
    finally:
        for L in dev + cached:
            k3.k3moe_layer_free(L)
        k3.k3moe_cache_destroy(cache)
