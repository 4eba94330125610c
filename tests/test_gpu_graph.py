"""Layer calls of a device-resident layer contain no host synchronisation, so they can be captured
in a CUDA graph and replayed with the eager calls' bytes: by a caller's stream capture (here
torch's), and by the library's own k3moe_graph_create / k3moe_graph_launch.  Covered: the
single-token decode path (fused router selection), a multi-unit decode call, the tensor-core GEMM
path, a residual + RMSNorm step between two captured layers, and the graph API's refusals."""
import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import mxfp4_routed_expert_06_b300 as k3  # noqa: E402

d, f, E, k = 512, 256, 64, 6


def _layer(seed, T_max, path):
    nib, scl = synth.experts(seed, 0, 0, E, d, f)
    Wr = synth.router_weights(seed, 0, E, d)
    L = k3.k3moe_pack_experts(k3.dims(d, f, E, k, T_max), nib, scl, 0, Wr)
    k3.k3moe_set_option(L, k3.K3MOE_OPT_PATH, path)
    return L


@pytest.mark.parametrize("T,path", [(1, "AUTO"), (40, "AUTO"), (300, "GEMM")])
def test_captured_calls_replay_the_eager_bytes(T, path):
    calls = 3
    L = _layer(41, T, getattr(k3, f"K3MOE_PATH_{path}"))
    try:
        x = torch.from_numpy(synth.tokens_bf16(41, 0, 0, calls * T, d).view(np.int16)).cuda()
        y = torch.zeros((calls * T, d), dtype=torch.float32, device="cuda")

        def run(stream):
            for c in range(calls):
                sl = slice(c * T, (c + 1) * T)
                k3.k3moe_layer_forward(L, x[sl], T, y[sl], stream)

        run(torch.cuda.current_stream())  # eager (also sets the kernels' shared-memory limits)
        torch.cuda.synchronize()
        y_eager = y.clone()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        with torch.cuda.graph(g, stream=s):
            run(torch.cuda.current_stream())
        for _ in range(2):
            y.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(y, y_eager), f"T={T} {path}: replay differs from the eager calls"
        k3.k3moe_sync(L)
    finally:
        k3.k3moe_layer_free(L)


def test_captured_two_layer_step_with_glue():
    T = 2
    L0, L1 = _layer(43, T, k3.K3MOE_PATH_AUTO), _layer(44, T, k3.K3MOE_PATH_AUTO)
    try:
        x = torch.from_numpy(synth.tokens_bf16(43, 0, 0, T, d).view(np.int16)).cuda()
        r = torch.empty_like(x)
        xn = torch.empty_like(x)
        y0 = torch.empty((T, d), dtype=torch.float32, device="cuda")
        y1 = torch.empty_like(y0)

        def step(stream):
            r.copy_(x)
            k3.k3moe_layer_forward(L0, x, T, y0, stream)
            k3.k3moe_residual_rmsnorm(y0, r, T, d, 1e-6, r, xn, stream)
            k3.k3moe_layer_forward(L1, xn, T, y1, stream)

        step(torch.cuda.current_stream())
        torch.cuda.synchronize()
        ref = (y0.clone(), y1.clone(), r.clone())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=torch.cuda.Stream()):
            step(torch.cuda.current_stream())
        for t in (y0, y1, r):
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y0, ref[0]) and torch.equal(y1, ref[1]) and torch.equal(r, ref[2])
    finally:
        k3.k3moe_layer_free(L0)
        k3.k3moe_layer_free(L1)


@pytest.mark.parametrize("T,path", [(1, "AUTO"), (40, "AUTO"), (300, "GEMM")])
def test_c_abi_graph_replays_the_eager_bytes(T, path):
    """k3moe_graph_create / k3moe_graph_launch: the library's own capture of repeated calls."""
    calls = 3
    L = _layer(47, T, getattr(k3, f"K3MOE_PATH_{path}"))
    g = None
    try:
        x = torch.from_numpy(synth.tokens_bf16(47, 0, 0, calls * T, d).view(np.int16)).cuda()
        y_eager = torch.empty((calls * T, d), dtype=torch.float32, device="cuda")
        for c in range(calls):
            sl = slice(c * T, (c + 1) * T)
            k3.k3moe_layer_forward(L, x[sl], T, y_eager[sl])
        y = torch.zeros_like(y_eager)
        g = k3.k3moe_graph_create(L, x, T, calls, y)  # runs the calls once, then captures them
        torch.cuda.synchronize()
        assert torch.equal(y, y_eager)
        for _ in range(2):
            y.zero_()
            k3.k3moe_graph_launch(g)
            k3.k3moe_sync(L)
            assert torch.equal(y, y_eager), f"T={T} {path}: replay differs from the eager calls"
    finally:
        if g is not None:
            k3.k3moe_graph_destroy(g)
        k3.k3moe_layer_free(L)


def test_c_abi_graph_refusals():
    T = 2
    L = _layer(49, T, k3.K3MOE_PATH_AUTO)
    x = torch.zeros((4 * T, d), dtype=torch.int16, device="cuda")
    y = torch.zeros((4 * T * d + 4,), dtype=torch.float32, device="cuda")
    try:
        for args, what in [((L, x, T, 0, y), "calls"), ((L, x, T + 1, 1, y), "T"),
                           ((L, x, T, 1, y[1:]), "aligned")]:
            with pytest.raises(k3.K3MoEError) as ei:
                k3.k3moe_graph_create(*args)
            assert ei.value.code == k3.K3MOE_ERR_INVALID_ARG and what in str(ei.value)
        k3.k3moe_profile(L, 1)
        with pytest.raises(k3.K3MoEError) as ei:
            k3.k3moe_graph_create(L, x, T, 1, y)
        assert ei.value.code == k3.K3MOE_ERR_INVALID_ARG
        k3.k3moe_profile(L, 0)
    finally:
        k3.k3moe_layer_free(L)
    nib, scl = synth.experts(49, 0, 0, E, d, f)
    eb = k3.k3moe_packed_expert_bytes(k3.dims(d, f, E, k, T))
    cache = k3.k3moe_cache_create(E * eb, eb)
    Lc = k3.k3moe_pack_experts(k3.dims(d, f, E, k, T), nib, scl, 0, synth.router_weights(49, 0, E, d), None, cache)
    try:
        with pytest.raises(k3.K3MoEError) as ei:
            k3.k3moe_graph_create(Lc, x, T, 1, y)
        assert ei.value.code == k3.K3MOE_ERR_UNSUPPORTED
    finally:
        k3.k3moe_layer_free(Lc)
        k3.k3moe_cache_destroy(cache)
