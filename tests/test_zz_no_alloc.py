"""The allocation-free router + top-k entry point agrees with the regular one and with the oracle.

k3moe_router_topk_noalloc serves callers that may not allocate device memory (for example
code inside a framework whose memory pool owns the GPU, where an extra cudaMalloc can fail or
synchronise the device).  It keeps its scratch in a fixed array inside the library, shared by
all calls.  Its GEMV sums in another order than the regular router, so expert ids are compared
exactly on gap-separated tokens and weights within 1e-5.  This file is collected last so that a
stop-at-first-failure run has already run every other test; it also passes on its own in a
fresh process.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import assert_routing_matches, gap_filtered_tokens

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import mxfp4_routed_expert_06_b300 as k3  # noqa: E402


def _dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def _layer_router(d, f, E, k, T, Wr, bias):
    """The regular entry point needs a layer (which allocates); experts are irrelevant to routing."""
    nb, sb = synth.expert_bytes(d, f)
    n_exp = np.zeros((E, nb), np.uint8)
    s_exp = np.full((E, sb), 127, np.uint8)
    return k3.k3moe_pack_experts(k3.dims(d, f, E, k, T), n_exp, s_exp, 0, Wr, bias)


def _both(layer, x, Wr_d, bias_d, T, d, E, k):
    xd = _dev(x)
    idx_ref = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w_ref = torch.empty((T, k), dtype=torch.float32, device="cuda")
    k3.k3moe_router_topk(layer, xd, T, idx_ref, w_ref)
    idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), -7.0, dtype=torch.float32, device="cuda")
    k3.k3moe_router_topk_noalloc(xd, Wr_d, bias_d, T, d, E, k, idx, w)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy(), idx_ref.cpu().numpy(), w_ref.cpu().numpy()


@pytest.mark.parametrize("d,f,E,k,T,hot", [
    (512, 256, 64, 6, 17, False),
    (7168, 1536, 896, 16, 64, True),     # K3 router shape; the regular one runs on the tensor cores
    (256, 128, 4096, 32, 16, False),     # T*E = 65536 (the scratch limit), k = 32 (a warp), no bias
])
def test_noalloc_router_matches_layer_router_and_oracle(d, f, E, k, T, hot):
    torch.cuda.set_device(0)
    bias = synth.hot_bias(4, 0, E, max(k, 2 * k), 2.0) if hot else None
    Wr = synth.router_weights(4, 0, E, d)
    layer = _layer_router(d, f, E, k, T, Wr, bias)
    Wr_d = _dev(Wr)
    bias_d = None if bias is None else _dev(bias)
    try:
        for call in range(2):  # two calls in a row share (and must clear) the scratch
            x, _ = gap_filtered_tokens(4, 0, 100 * call, T, d, Wr, bias, k)
            idx, w, idx_ref, w_ref = _both(layer, x, Wr_d, bias_d, T, d, E, k)
            i_o, w_o, _, keys_o = oracle.router(x, Wr, bias, k)
            # against the regular entry point: the same expert sets, the same slot order wherever
            # the keys are separated, weights within 1e-5 (matched by expert id)
            assert_routing_matches(idx, w, idx_ref, w_ref, keys_o)
            assert_routing_matches(idx, w, i_o, w_o, keys_o)
    finally:
        k3.k3moe_layer_free(layer)


def test_noalloc_minus_inf_bias_keeps_ids_in_range():
    # A -inf bias masks E-k+1 experts, so only k-1 keys are finite: the k-th pick is the
    # lowest-id masked expert (equal keys, lower id first), never an out-of-range id.
    d, f, E, k, T = 512, 256, 64, 8, 5
    Wr = synth.router_weights(6, 0, E, d)
    bias = np.full(E, -np.inf, np.float32)
    open_ = np.array([3, 9, 17, 30, 41, 50, 62])  # k - 1 experts stay selectable
    bias[open_] = 0.0
    layer = _layer_router(d, f, E, k, T, Wr, bias)
    try:
        x = synth.tokens_bf16(6, 0, 0, T, d)
        idx, w, idx_ref, w_ref = _both(layer, x, _dev(Wr), _dev(bias), T, d, E, k)
        assert idx.min() >= 0 and idx.max() < E
        i_o, w_o, _, keys_o = oracle.router(x, Wr, bias, k)
        masked_first = int(np.setdiff1d(np.arange(E), open_)[0])
        for t in range(T):
            assert sorted(idx[t, :k - 1].tolist()) == sorted(open_.tolist())
            assert idx[t, k - 1] == masked_first
            assert sorted(idx[t].tolist()) == sorted(idx_ref[t].tolist()) == sorted(i_o[t].tolist())
        np.testing.assert_allclose(w, w_ref, rtol=0, atol=1e-5)
        assert_routing_matches(idx, w, i_o, w_o, keys_o)
    finally:
        k3.k3moe_layer_free(layer)


def test_noalloc_rejects_oversized_request():
    d, E, k, T = 256, 4096, 4, 17  # T*E = 69632 > 65536
    x = torch.zeros((T, d), dtype=torch.int16, device="cuda")
    Wr = torch.zeros((E, d), dtype=torch.float32, device="cuda")
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    with pytest.raises(k3.K3MoEError) as ei:
        k3.k3moe_router_topk_noalloc(x, Wr, None, T, d, E, k, idx, w)
    assert ei.value.code == k3.K3MOE_ERR_INVALID_ARG and "65536" in str(ei.value)
