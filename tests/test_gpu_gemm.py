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
    128 picks per hot expert on average.  Sampled tokens against the oracle; all tokens against
    the register-decode path."""
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
    rel = np.linalg.norm(y_g - y_d, axis=1) / np.linalg.norm(y_d, axis=1)
    assert rel.max() < 2e-3, rel.max()
    for t in (0, 117, T - 1):
        idx_o, w_o, _, keys = oracle.router(x[t:t + 1], Wr, bias, k)
        assert set(idx_o[0].tolist()) <= set(np.nonzero(bias)[0].tolist())
        nibs, scls = [], []
        for e in idx_o[0].tolist():
            n_, s_ = synth.experts(41, 0, e, e + 1, d, f)
            nibs.append(n_[0])
            scls.append(s_[0])
        y_o, sumabs = oracle.moe(x[t:t + 1], w_o, nibs, scls, f)
        assert_y_close(y_g[t:t + 1], y_o, sumabs, f"K3 gemm token {t}")
    k3.k3moe_layer_free(L)
