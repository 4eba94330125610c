"""Edge cases of the layer against the fp64 oracle: the degenerate routings (every expert
picked, a single expert), the largest k, E and d the boundary accepts, and T = T_max through
both FFN paths.  Routing and bucketing must match exactly, y within 2e-3 * sum|terms| + 1e-5."""
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


def _run(L, x, T, d, k, path):
    k3.k3moe_set_option(L, k3.K3MOE_OPT_PATH, path)
    xd = _dev(x)
    y = torch.empty((T, d), dtype=torch.float32, device="cuda")
    k3.k3moe_layer_forward(L, xd, T, y)
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    k3.k3moe_router_topk(L, xd, T, idx, w)
    k3.k3moe_sync(L)
    return y.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("d,f,E,k,T", [
    (256, 128, 4, 4, 5),       # k = E: every expert is picked, weights are the normalised sigmoids
    (128, 128, 1, 1, 3),       # a single expert: w = 1, y = the expert's output
    (256, 128, 64, 32, 9),     # the largest k
    (128, 128, 4096, 8, 6),    # the largest E
    (16384, 128, 4, 2, 3),     # the largest d
])
@pytest.mark.parametrize("path", ["decode", "gemm"])
def test_boundary_shapes(d, f, E, k, T, path):
    seed = 61
    nib, scl = synth.experts(seed, 0, 0, E, d, f)
    Wr = synth.router_weights(seed, 0, E, d)
    L = k3.k3moe_pack_experts(k3.dims(d, f, E, k, T), nib, scl, 0, Wr)
    x, _ = gap_filtered_tokens(seed, 0, 0, T, d, Wr, None, k)
    ref = oracle.layer(x, Wr, None, k, f, nib, scl)
    p = k3.K3MOE_PATH_DECODE if path == "decode" else k3.K3MOE_PATH_GEMM
    y, idx, w = _run(L, x, T, d, k, p)
    assert_routing_matches(idx, w, ref["idx"], ref["w"], ref["keys"])
    if k == E:
        assert np.allclose(w.sum(axis=1), 1.0, atol=1e-6)
    assert_y_close(y, ref["y"], ref["sumabs"], f"{path} d={d} f={f} E={E} k={k} T={T}")
    k3.k3moe_layer_free(L)


@pytest.mark.parametrize("path", ["decode", "gemm"])
def test_t_max(path):
    """T = T_max = 65536 tokens on a small layer: routing and bucketing of every token, y of
    sampled tokens (first, last and a seeded sample)."""
    d, f, E, k, T = 128, 128, 8, 2, 65536
    seed = 67
    nib, scl = synth.experts(seed, 0, 0, E, d, f)
    Wr = synth.router_weights(seed, 0, E, d)
    L = k3.k3moe_pack_experts(k3.dims(d, f, E, k, T), nib, scl, 0, Wr)
    x, _ = gap_filtered_tokens(seed, 0, 0, T, d, Wr, None, k)
    p = k3.K3MOE_PATH_DECODE if path == "decode" else k3.K3MOE_PATH_GEMM
    y, idx, w = _run(L, x, T, d, k, p)
    idx_o, w_o, _, keys = oracle.router(x, Wr, None, k)
    assert_routing_matches(idx, w, idx_o, w_o, keys)
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * k, dtype=torch.int32, device="cuda")
    k3.k3moe_bucket(L, _dev(idx), T, counts, offsets, perm)
    torch.cuda.synchronize()
    c_o, o_o, p_o = oracle.bucket(idx_o, E)
    assert np.array_equal(counts.cpu().numpy(), c_o)
    assert np.array_equal(offsets.cpu().numpy(), o_o)
    assert np.array_equal(perm.cpu().numpy(), p_o)
    rng = np.random.default_rng(5)
    sample = np.unique(np.concatenate([[0, T - 1], rng.choice(T, 30, replace=False)]))
    xs = x[sample]
    ref = oracle.layer(xs, Wr, None, k, f, nib, scl)
    assert_y_close(y[sample], ref["y"], ref["sumabs"], f"{path} T={T}")
    k3.k3moe_layer_free(L)
