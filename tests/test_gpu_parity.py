"""Parity of the CUDA path (through the C ABI) against the fp64 CPU oracle.

Routing (top-k sets) and bucketing must match exactly; y must be within
2e-3 * sum|terms| + 1e-5 per element (the bound the layer's accuracy target states).
Small configurations span several tiles and ragged token counts; the full Kimi K3
shape (d=7168, f=1536, E=896, k=16) is checked on sampled tokens.
"""
import os

import numpy as np
import pytest

import oracle
import synth
from helpers import (GAP_MIN, assert_routing_matches, assert_routing_valid, assert_y_close, gap_filtered_tokens,
                     unpack_tiles)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import mxfp4_routed_expert_06_b300 as k3  # noqa: E402


def _dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


class Small:
    """A layer small enough that the oracle runs it whole."""

    def __init__(self, d, f, E, k, T_max, seed=1, bias=None, scale_lo=121, scale_hi=125, nib=None, scl=None):
        self.d, self.f, self.E, self.k = d, f, E, k
        self.seed = seed
        if nib is None:
            nib, scl = synth.experts(seed, 0, 0, E, d, f, scale_lo, scale_hi)
        self.nib, self.scl = nib, scl
        self.Wr = synth.router_weights(seed, 0, E, d)
        self.bias = bias
        self.layer = k3.k3moe_pack_experts(k3.dims(d, f, E, k, T_max), nib, scl, 0, self.Wr, bias)

    def tokens(self, T, t0=0):
        x, _ = gap_filtered_tokens(self.seed, 0, t0, T, self.d, self.Wr, self.bias, self.k)
        return x

    def forward(self, x):
        T = x.shape[0]
        y = torch.empty((T, self.d), dtype=torch.float32, device="cuda")
        k3.k3moe_layer_forward(self.layer, _dev(x), T, y)
        torch.cuda.synchronize()
        return y.cpu().numpy()

    def routing(self, x):
        T = x.shape[0]
        idx = torch.empty((T, self.k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, self.k), dtype=torch.float32, device="cuda")
        k3.k3moe_router_topk(self.layer, _dev(x), T, idx, w)
        torch.cuda.synchronize()
        return idx.cpu().numpy(), w.cpu().numpy()

    def free(self):
        k3.k3moe_layer_free(self.layer)


def _check_layer(L: Small, x, what):
    ref = oracle.layer(x, L.Wr, L.bias, L.k, L.f, L.nib, L.scl)
    idx, w = L.routing(x)
    assert_routing_matches(idx, w, ref["idx"], ref["w"], ref["keys"])
    y = L.forward(x)
    return assert_y_close(y, ref["y"], ref["sumabs"], what)


def test_device_generator_matches_host():
    for d, f, e0, e1 in [(256, 128, 0, 3), (7168, 1536, 895, 896)]:
        nb, sb = synth.expert_bytes(d, f)
        n = e1 - e0
        dn = torch.empty(n * nb, dtype=torch.uint8, device="cuda")
        ds = torch.empty(n * sb, dtype=torch.uint8, device="cuda")
        synth.experts_to_device(7, 2, e0, e1, d, f, dn.data_ptr(), ds.data_ptr())
        torch.cuda.synchronize()
        hn, hs = synth.experts(7, 2, e0, e1, d, f)
        assert np.array_equal(dn.cpu().numpy(), hn.reshape(-1))
        assert np.array_equal(ds.cpu().numpy(), hs.reshape(-1))


def test_pack_layout_round_trip():
    L = Small(256, 128, 8, 2, 4)
    nb = k3.k3moe_packed_expert_bytes(k3.dims(256, 128, 8, 2, 4))
    for e in range(8):
        buf = np.empty(nb, np.uint8)
        k3.k3moe_read_packed(L.layer, e, buf)
        n, s = unpack_tiles(buf, 256, 128)
        assert np.array_equal(n, L.nib[e]) and np.array_equal(s, L.scl[e])
    L.free()


def test_tiny_config_c1():
    # d=256, f=128, E=8, k=2, T=4, no bias: the smallest configuration, run whole.
    L = Small(256, 128, 8, 2, 4)
    x = L.tokens(4)
    ref = oracle.layer(x, L.Wr, None, 2, 128, L.nib, L.scl)
    idx, w = L.routing(x)
    assert_routing_matches(idx, w, ref["idx"], ref["w"], ref["keys"])
    # bucketing entry point on the same picks
    counts = torch.empty(8, dtype=torch.int32, device="cuda")
    offsets = torch.empty(9, dtype=torch.int32, device="cuda")
    perm = torch.empty(8, dtype=torch.int32, device="cuda")
    k3.k3moe_bucket(L.layer, _dev(idx), 4, counts, offsets, perm)
    torch.cuda.synchronize()
    c_o, o_o, p_o = oracle.bucket(idx, 8)
    assert counts.cpu().numpy().tolist() == c_o.tolist()
    assert offsets.cpu().numpy().tolist() == o_o.tolist()
    assert perm.cpu().numpy().tolist() == p_o.tolist()
    y = L.forward(x)
    assert_y_close(y, ref["y"], ref["sumabs"], "C1")
    L.free()


@pytest.mark.parametrize("d,f,E,k,T", [
    (512, 256, 16, 4, 1),
    (512, 256, 16, 4, 3),
    (384, 384, 32, 8, 17),
    (1024, 512, 64, 6, 64),
    (384, 128, 12, 3, 129),
    (512, 256, 40, 9, 120),   # 1080 picks: separate top-k and bucketing kernels
    (256, 128, 64, 32, 1),    # 32 picks (k = 32): the one-warp fused bucketing at its limit
    (256, 256, 24, 16, 2),    # 32 picks (k = 16, T = 2)
    (256, 128, 48, 11, 3),    # 33 picks: the block-wide fused bucketing
])
def test_small_configs(d, f, E, k, T):
    L = Small(d, f, E, k, T, seed=d + f + E + k + T)
    _check_layer(L, L.tokens(T), f"d{d} f{f} E{E} k{k} T{T}")
    L.free()


def test_bias_steers_selection_hot_expert():
    # a +10 bias on expert 3 with k=1: every token picks expert 3 (40 tokens > 8 per pass),
    # and its combine weight is 1 (sigmoid of the unbiased logit, renormalised).
    d, f, E = 256, 128, 8
    bias = np.zeros(E, np.float32)
    bias[3] = 10.0
    L = Small(d, f, E, 1, 40, seed=5, bias=bias)
    x = L.tokens(40)
    idx, w = L.routing(x)
    assert np.all(idx == 3) and np.all(w == 1.0)
    _check_layer(L, x, "hot expert")
    L.free()


def test_hot_subset_bias_k3():
    d, f, E, k = 512, 256, 24, 4
    bias = synth.hot_bias(9, 0, E, 6, 2.0)
    L = Small(d, f, E, k, 33, seed=9, bias=bias)
    x = L.tokens(33)
    idx, _ = L.routing(x)
    assert set(np.unique(idx)) <= set(np.nonzero(bias)[0].tolist())
    _check_layer(L, x, "hot subset")
    L.free()


def test_zero_nibbles_give_zero_output():
    d, f, E, k = 256, 128, 8, 2
    nb, sb = synth.expert_bytes(d, f)
    nib = np.zeros((E, nb), np.uint8)
    nib[:, : nb // 3] = 0x88  # gate all -0
    scl = np.full((E, sb), 123, np.uint8)
    L = Small(d, f, E, k, 5, nib=nib, scl=scl)
    y = L.forward(L.tokens(5))
    assert np.all(y == 0)
    L.free()


@pytest.mark.parametrize("lo,hi", [(121, 121), (125, 125), (110, 135)])
def test_scale_extremes(lo, hi):
    L = Small(256, 256, 8, 2, 6, seed=lo * hi, scale_lo=lo, scale_hi=hi)
    _check_layer(L, L.tokens(6), f"scales {lo}..{hi}")
    L.free()


def test_nan_scale_refused():
    d, f, E = 256, 128, 4
    nib, scl = synth.experts(1, 0, 0, E, d, f)
    scl[2, 17] = 255
    Wr = synth.router_weights(1, 0, E, d)
    with pytest.raises(k3.K3MoEError) as ei:
        k3.k3moe_pack_experts(k3.dims(d, f, E, 2, 4), nib, scl, 0, Wr)
    assert ei.value.code == k3.K3MOE_ERR_INVALID_ARG


def test_bucket_entry_point_large():
    E, k, T = 64, 8, 300
    L = Small(256, 128, E, k, T)
    rng = np.random.default_rng(3)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * k, dtype=torch.int32, device="cuda")
    k3.k3moe_bucket(L.layer, _dev(idx), T, counts, offsets, perm)
    torch.cuda.synchronize()
    c_o, o_o, p_o = oracle.bucket(idx, E)
    assert np.array_equal(counts.cpu().numpy(), c_o)
    assert np.array_equal(offsets.cpu().numpy(), o_o)
    assert np.array_equal(perm.cpu().numpy(), p_o)
    L.free()


@pytest.mark.parametrize("E,k,T", [
    (896, 16, 300),    # 4800 picks: chunks of 2048 with a ragged last one (multi-CTA bucketing)
    (1536, 8, 700),    # the largest E the multi-CTA scatter keeps its per-warp histograms for
    (2048, 4, 1100),   # larger E: the single-block kernel
])
def test_bucket_entry_point_many_picks(E, k, T):
    L = Small(256, 128, E, k, T)
    rng = np.random.default_rng(E + T)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * k, dtype=torch.int32, device="cuda")
    for _ in range(2):  # the per-chunk scratch is rewritten each call
        k3.k3moe_bucket(L.layer, _dev(idx), T, counts, offsets, perm)
        torch.cuda.synchronize()
        c_o, o_o, p_o = oracle.bucket(idx, E)
        assert np.array_equal(counts.cpu().numpy(), c_o)
        assert np.array_equal(offsets.cpu().numpy(), o_o)
        assert np.array_equal(perm.cpu().numpy(), p_o)
    L.free()


def test_deterministic_and_host_entry_point():
    L = Small(512, 256, 16, 4, 9)
    x = L.tokens(9)
    y1 = L.forward(x)
    y2 = L.forward(x)
    assert np.array_equal(y1, y2)
    yh = np.empty((9, 512), np.float32)  # pageable: staging buffer and a copy back
    k3.k3moe_layer_forward_host(L.layer, np.ascontiguousarray(x), 9, yh)
    assert np.array_equal(yh, y1)
    # pinned host memory, aligned or 4 bytes off a 16-byte boundary (staging buffers hold x and y)
    pin = torch.zeros(9 * 512 + 4, dtype=torch.float32).pin_memory()
    for off in (0, 1):
        yp = pin[off:off + 9 * 512].view(9, 512)
        yp.zero_()
        k3.k3moe_layer_forward_host(L.layer, np.ascontiguousarray(x), 9, yp)
        assert np.array_equal(yp.numpy(), y1), f"pinned y_host at float offset {off}"
    # a device y that is not 16-byte aligned is refused before any work is queued
    yd = torch.zeros(9 * 512 + 4, dtype=torch.float32, device="cuda")
    xd = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda()
    with pytest.raises(k3.K3MoEError) as ei:
        k3.k3moe_layer_forward(L.layer, xd, 9, yd[1:1 + 9 * 512])
    assert ei.value.code == k3.K3MOE_ERR_INVALID_ARG and "y must be 16-byte aligned" in str(ei.value)
    # int32 / float32 outputs 2 bytes off their natural alignment: refused, nothing queued
    buf = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    p0 = buf.data_ptr()
    h = k3._handle(L.layer)
    assert k3._lib.k3moe_router_topk(h, xd.data_ptr(), 9, p0 + 2, p0 + 1024, None) == k3.K3MOE_ERR_INVALID_ARG
    assert k3._lib.k3moe_router_topk(h, xd.data_ptr(), 9, p0, p0 + 1026, None) == k3.K3MOE_ERR_INVALID_ARG
    assert k3._lib.k3moe_bucket(h, p0 + 2, 9, p0 + 1024, p0 + 2048, p0 + 3072, None) == k3.K3MOE_ERR_INVALID_ARG
    assert k3._lib.k3moe_bucket(h, p0, 9, p0 + 1024, p0 + 2050, p0 + 3072, None) == k3.K3MOE_ERR_INVALID_ARG
    assert "aligned" in k3._lib.k3moe_last_error().decode()
    torch.cuda.synchronize()
    L.free()


# ------------------------------------------------------------------ Kimi K3 shape ---

K3D, K3F, K3E, K3K = 7168, 1536, 896, 16
SEED = 2026


@pytest.fixture(scope="module")
def k3_layer():
    """One full K3-shaped layer: 896 experts generated on the device, packed, 15.7 GB resident."""
    nb, sb = synth.expert_bytes(K3D, K3F)
    dn = torch.empty(K3E * nb, dtype=torch.uint8, device="cuda")
    ds = torch.empty(K3E * sb, dtype=torch.uint8, device="cuda")
    synth.experts_to_device(SEED, 0, 0, K3E, K3D, K3F, dn.data_ptr(), ds.data_ptr())
    Wr = synth.router_weights(SEED, 0, K3E, K3D)
    layer = k3.k3moe_pack_experts(k3.dims(K3D, K3F, K3E, K3K, 64), dn, ds, 1, _dev(Wr), None)
    del dn, ds
    torch.cuda.empty_cache()
    yield layer, Wr
    k3.k3moe_layer_free(layer)


def _k3_oracle_y(x, idx, w):
    """Oracle y for K3-shaped tokens; the experts are regenerated on the host one by one."""
    cache = {}
    nibs, scls = [], []
    for e in idx.reshape(-1).tolist():
        if e not in cache:
            n, s = synth.experts(SEED, 0, e, e + 1, K3D, K3F)
            cache[e] = (n[0], s[0])
        nibs.append(cache[e][0])
        scls.append(cache[e][1])
    return oracle.moe(x, w, nibs, scls, K3F)


def _run(layer, x):
    T = x.shape[0]
    y = torch.empty((T, K3D), dtype=torch.float32, device="cuda")
    idx = torch.empty((T, K3K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, K3K), dtype=torch.float32, device="cuda")
    k3.k3moe_router_topk(layer, _dev(x), T, idx, w)
    k3.k3moe_layer_forward(layer, _dev(x), T, y)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy(), y.cpu().numpy()


def test_k3_single_token_decode(k3_layer):
    # the single-token decode workload: T = 1 calls, as the benchmark times them
    layer, Wr = k3_layer
    x, _ = gap_filtered_tokens(SEED, 0, 0, 3, K3D, Wr, None, K3K)
    for t in range(3):
        xt = x[t:t + 1]
        idx, w, y = _run(layer, xt)
        i_o, w_o, _, keys = oracle.router(xt, Wr, None, K3K)
        assert_routing_matches(idx, w, i_o, w_o, keys)
        y_o, sa = _k3_oracle_y(xt, i_o, w_o)
        assert_y_close(y, y_o, sa, f"K3 T=1 token {t}")


def test_k3_batched_decode_t64(k3_layer):
    layer, Wr = k3_layer
    T = 64
    x, _ = gap_filtered_tokens(SEED, 0, 1000, T, K3D, Wr, None, K3K)
    idx, w, y = _run(layer, x)
    i_o, w_o, _, keys = oracle.router(x, Wr, None, K3K)
    assert_routing_matches(idx, w, i_o, w_o, keys)
    # bucketing of all 1024 picks, exact
    counts = torch.empty(K3E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(K3E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * K3K, dtype=torch.int32, device="cuda")
    k3.k3moe_bucket(layer, _dev(idx), T, counts, offsets, perm)
    torch.cuda.synchronize()
    c_o, o_o, p_o = oracle.bucket(idx, K3E)
    assert np.array_equal(counts.cpu().numpy(), c_o) and np.array_equal(perm.cpu().numpy(), p_o)
    assert np.array_equal(offsets.cpu().numpy(), o_o)
    # y on every token of the batch, element by element
    y_o, sa = _k3_oracle_y(x, i_o, w_o)
    assert_y_close(y, y_o, sa, "K3 T=64, all tokens")
    # whole-batch invariant at any size: bitwise repeatable
    _, _, y2 = _run(layer, x)
    assert np.array_equal(y, y2)


def _bench_check(layer, Wr, x, T, calls, n_y, what):
    """The benchmark's own tokens (its seed and stream offset, no gap filter) in its launch
    configuration: `calls` layer calls of T tokens.  Routing of every token against the oracle:
    exact where the oracle's k-th/(k+1)-th key gap is at least GAP_MIN, a valid top-k within the
    router's rounding elsewhere.  y of n_y sampled separated tokens (first and last included)
    element by element against the oracle.  A second pass over all calls is bitwise identical."""
    n = T * calls
    xd = _dev(x)
    idx = torch.empty((n, K3K), dtype=torch.int32, device="cuda")
    w = torch.empty((n, K3K), dtype=torch.float32, device="cuda")
    ys = [torch.empty((n, K3D), dtype=torch.float32, device="cuda") for _ in range(2)]
    for c in range(calls):
        sl = slice(c * T, (c + 1) * T)
        k3.k3moe_router_topk(layer, xd[sl], T, idx[sl], w[sl])
    for y in ys:
        for c in range(calls):
            sl = slice(c * T, (c + 1) * T)
            k3.k3moe_layer_forward(layer, xd[sl], T, y[sl])
    torch.cuda.synchronize()
    assert torch.equal(ys[0], ys[1]), f"{what}: not bitwise repeatable"
    idx_h, w_h, y_h = idx.cpu().numpy(), w.cpu().numpy(), ys[0].cpu().numpy()
    i_o, w_o, lg_o, keys = oracle.router(x, Wr, None, K3K)
    sep = oracle.topk_gap(keys, K3K) >= GAP_MIN
    assert sep.sum() >= n // 2
    assert_routing_matches(idx_h[sep], w_h[sep], i_o[sep], w_o[sep], keys[sep])
    # fp32 GEMV (T < 64) or bf16 hi+lo tensor-core logits (T >= 64, error <= 4e-4 worst case)
    assert_routing_valid(idx_h[~sep], w_h[~sep], lg_o[~sep], keys[~sep], 1e-5 if T < 64 else 5e-4)
    cand = np.nonzero(sep)[0]
    rng = np.random.default_rng(SEED + T)
    sample = sorted(set(rng.choice(cand[1:-1], size=n_y - 2, replace=False).tolist()) | {int(cand[0]), int(cand[-1])})
    y_o, sa = _k3_oracle_y(x[sample], i_o[sample], w_o[sample])
    assert_y_close(y_h[sample], y_o, sa, f"{what}, {len(sample)} sampled tokens")


def test_k3_benchmark_tokens_single_token_decode(k3_layer):
    """The single-token decode benchmark's 1000 tokens, one T=1 call each."""
    layer, Wr = k3_layer
    x = synth.tokens_bf16(SEED, 0, 0, 1000, K3D)
    _bench_check(layer, Wr, x, 1, 1000, 24, "K3 T=1 benchmark tokens")


@pytest.mark.skipif(os.environ.get("K3MOE_ORACLE_ALL") != "1",
                    reason="opt-in (K3MOE_ORACLE_ALL=1): every token through the oracle, about 10 minutes each")
@pytest.mark.parametrize("T,calls,t0", [(1, 1000, 0), (64, 15, 1_000_000)])
def test_k3_benchmark_tokens_every_output(k3_layer, T, calls, t0):
    """A decode benchmark's own tokens (single-token: 1000 calls; batched: 15 calls of 64), every y
    element against the oracle.  A token whose 16th/17th oracle keys lie within GAP_MIN is checked
    on the GPU's own picks (a valid top-k, checked as such) with the oracle's fp64 weights for them;
    the others on the oracle's routing."""
    layer, Wr = k3_layer
    n = T * calls
    x = synth.tokens_bf16(SEED, 0, t0, n, K3D)
    xd = _dev(x)
    y = torch.empty((n, K3D), dtype=torch.float32, device="cuda")
    idx = torch.empty((n, K3K), dtype=torch.int32, device="cuda")
    w = torch.empty((n, K3K), dtype=torch.float32, device="cuda")
    for c in range(calls):
        sl = slice(c * T, (c + 1) * T)
        k3.k3moe_router_topk(layer, xd[sl], T, idx[sl], w[sl])
        k3.k3moe_layer_forward(layer, xd[sl], T, y[sl])
    torch.cuda.synchronize()
    y_h, idx_h, w_h = y.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()
    i_o, w_o, lg_o, keys = oracle.router(x, Wr, None, K3K)
    sep = oracle.topk_gap(keys, K3K) >= GAP_MIN
    assert_routing_matches(idx_h[sep], w_h[sep], i_o[sep], w_o[sep], keys[sep])
    assert_routing_valid(idx_h[~sep], w_h[~sep], lg_o[~sep], keys[~sep], 1e-5 if T < 64 else 5e-4)
    # the picks each token is checked on, with fp64 weights for them
    sig = 1.0 / (1.0 + np.exp(-lg_o))
    picks = np.where(sep[:, None], i_o, idx_h)
    wts = np.take_along_axis(sig, picks.astype(np.int64), axis=1)
    wts = wts / wts.sum(axis=1, keepdims=True)
    cache = {}
    for b0 in range(0, n, 50):
        ts = np.arange(b0, min(n, b0 + 50))
        nibs, scls = [], []
        for e in picks[ts].reshape(-1).tolist():
            if e not in cache:
                n_, s_ = synth.experts(SEED, 0, e, e + 1, K3D, K3F)
                cache[e] = (n_[0], s_[0])
            nibs.append(cache[e][0])
            scls.append(cache[e][1])
        y_o, sa = oracle.moe(x[ts], wts[ts], nibs, scls, K3F)
        assert_y_close(y_h[ts], y_o, sa, f"K3 T={T} benchmark tokens {b0}..{ts[-1]}")


def test_k3_benchmark_tokens_batched_decode(k3_layer):
    """The batched decode benchmark's 15 calls of 64 tokens (its stream offset in the default run)."""
    layer, Wr = k3_layer
    x = synth.tokens_bf16(SEED, 0, 1_000_000, 15 * 64, K3D)
    _bench_check(layer, Wr, x, 64, 15, 16, "K3 T=64 benchmark tokens")


def test_bounded_wait_reports_timeout_and_context_survives():
    # A forward whose FFN consumers wait on a barrier that nothing completes: the bounded wait
    # (50 ms here) gives up, the kernels return, k3moe_sync reports the timeout, and the next
    # call on the same context is correct.  No GPU fault or hang is involved.
    L = Small(256, 128, 8, 2, 4)
    x = L.tokens(4)
    y_ok = L.forward(x)
    k3.k3moe_sync(L.layer)
    k3.k3moe_set_option(L.layer, k3.K3MOE_OPT_DEVICE_WAIT_NS, 50_000_000)
    k3.k3moe_set_option(L.layer, k3.K3MOE_OPT_TEST_STALL, 1)
    y = torch.empty((4, 256), dtype=torch.float32, device="cuda")
    k3.k3moe_layer_forward(L.layer, _dev(x), 4, y)
    with pytest.raises(k3.K3MoEError) as ei:
        k3.k3moe_sync(L.layer)
    assert ei.value.code == k3.K3MOE_ERR_TIMEOUT
    assert np.array_equal(L.forward(x), y_ok)
    k3.k3moe_sync(L.layer)
    L.free()


def test_zero_scale_bytes():
    # E8M0 byte 0 is 2^-127 (a subnormal in fp32): the layer is flagged at pack time and the
    # kernels take the exact decode for it.
    d, f, E, k = 256, 256, 8, 2
    nib, scl = synth.experts(3, 0, 0, E, d, f)
    scl[:, ::7] = 0
    L = Small(d, f, E, k, 6, seed=3, nib=nib, scl=scl)
    _check_layer(L, L.tokens(6), "zero scales")
    L.free()


@pytest.mark.parametrize("path,T", [("decode", 5), ("decode", 40), ("gemm", 300)])
def test_situ_glu_option_matches_oracle(path, T):
    # K3MOE_OPT_ACTIVATION = SiTU-GLU (a reading of the deep dive's glossary entry; the oracle
    # restates the same reading): both FFN paths against the oracle, and the option takes effect.
    d, f, E, k = 512, 256, 16, 4
    L = Small(d, f, E, k, T, seed=77 + T)
    x = L.tokens(T)
    k3.k3moe_set_option(L.layer, k3.K3MOE_OPT_PATH, k3.K3MOE_PATH_GEMM if path == "gemm" else k3.K3MOE_PATH_DECODE)
    y_swiglu = L.forward(x)
    k3.k3moe_set_option(L.layer, k3.K3MOE_OPT_ACTIVATION, k3.K3MOE_ACT_SITU_GLU)
    y = L.forward(x)
    ref = oracle.layer(x, L.Wr, None, k, f, L.nib, L.scl, act=oracle.ACT_SITU_GLU)
    assert_y_close(y, ref["y"], ref["sumabs"], f"SiTU-GLU, {path} path, T={T}")
    assert not np.allclose(y, y_swiglu)
    assert np.array_equal(L.forward(x), y)  # deterministic
    with pytest.raises(k3.K3MoEError):
        k3.k3moe_set_option(L.layer, k3.K3MOE_OPT_ACTIVATION, 7)
    L.free()


@pytest.mark.parametrize("src_on_device,cached", [(0, False), (1, False), (0, True)])
def test_layer_from_saved_packed_pool_is_byte_identical(src_on_device, cached):
    # a packed pool saved with its header (k3moe_read_packed per expert + k3moe_pool_header_get)
    # loads into a new layer without repacking and gives the original layer's bytes
    d, f, E, k, T = 512, 256, 16, 4, 6
    L = Small(d, f, E, k, T, seed=91)
    dm = k3.dims(d, f, E, k, T)
    eb = k3.k3moe_packed_expert_bytes(dm)
    hdr = k3.k3moe_pool_header_get(L.layer)
    k3.k3moe_pool_header_check(hdr, dm)
    assert (hdr.s_min, hdr.s_max, hdr.expert_bytes) == (int(L.scl.min()), int(L.scl.max()), eb)
    pool = np.empty(E * eb, np.uint8)
    for e in range(E):
        k3.k3moe_read_packed(L.layer, e, pool[e * eb:(e + 1) * eb])
    src = torch.from_numpy(pool).cuda() if src_on_device else pool
    Wr = _dev(L.Wr) if src_on_device else L.Wr
    cache = k3.k3moe_cache_create(E * eb, eb) if cached else None
    L2 = k3.k3moe_layer_from_packed(dm, hdr, src, src_on_device, Wr, None, cache)
    try:
        x = L.tokens(T)
        y = torch.empty((T, d), dtype=torch.float32, device="cuda")
        k3.k3moe_layer_forward(L2, _dev(x), T, y)
        torch.cuda.synchronize()
        assert np.array_equal(y.cpu().numpy(), L.forward(x))
        bad = k3.k3moe_pool_header_get(L.layer)
        bad.E = 15
        with pytest.raises(k3.K3MoEError):
            k3.k3moe_layer_from_packed(dm, bad, src, src_on_device, Wr)
    finally:
        k3.k3moe_layer_free(L2)
        if cache is not None:
            k3.k3moe_cache_destroy(cache)
        L.free()
