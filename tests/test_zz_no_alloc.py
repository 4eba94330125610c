"""The allocation-free router + top-k entry point agrees with the regular one.

k3moe_router_topk_noalloc serves callers that may not allocate device memory (for example
code inside a framework whose memory pool owns the GPU, where an extra cudaMalloc can fail or
synchronise the device).  It keeps its scratch in a fixed array inside the library, shared by
all calls.  This file is collected last so that a stop-at-first-failure run has already run
every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import mxfp4_routed_expert_06_b300 as k3  # noqa: E402


def _dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


@pytest.mark.parametrize("d,f,E,k,T,hot", [(512, 256, 64, 6, 17, False), (7168, 1536, 896, 16, 64, True)])
def test_noalloc_router_matches_layer_router(d, f, E, k, T, hot):
    torch.cuda.set_device(0)
    bias = synth.hot_bias(4, 0, E, max(k, 2 * k), 2.0) if hot else None
    Wr = synth.router_weights(4, 0, E, d)
    nb, sb = synth.expert_bytes(d, f)
    # the regular entry point needs a layer (which allocates); experts are irrelevant to routing
    n_exp = np.zeros((E, nb), np.uint8)
    s_exp = np.full((E, sb), 127, np.uint8)
    layer = k3.k3moe_pack_experts(k3.dims(d, f, E, k, T), n_exp, s_exp, 0, Wr, bias)
    Wr_d = _dev(Wr)
    bias_d = None if bias is None else _dev(bias)
    try:
        for call in range(2):  # two calls in a row share (and must clear) the scratch
            x = _dev(synth.tokens_bf16(4, 0, 100 * call, T, d))
            idx_ref = torch.empty((T, k), dtype=torch.int32, device="cuda")
            w_ref = torch.empty((T, k), dtype=torch.float32, device="cuda")
            k3.k3moe_router_topk(layer, x, T, idx_ref, w_ref)
            idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
            w = torch.full((T, k), -7.0, dtype=torch.float32, device="cuda")
            k3.k3moe_router_topk_noalloc(x, Wr_d, bias_d, T, d, E, k, idx, w)
            torch.cuda.synchronize()
            assert torch.equal(idx, idx_ref), f"call {call}: expert ids differ"
            # from 64 tokens the regular entry point computes the logits on the tensor cores
            # (W_r split into bf16 hi + lo), so the weights agree to the bound the oracle
            # comparisons use, not bitwise
            np.testing.assert_allclose(w.cpu().numpy(), w_ref.cpu().numpy(), rtol=0, atol=1e-5)
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
