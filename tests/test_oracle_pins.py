"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test ties one oracle function to a value the pages print, a hand-worked
example, a closed form, an invariant, brute force, or a library routine used as
an independent second formulation.  A plausible slip in the oracle (a wrong
nibble order, a transposed matrix, a dropped bias, weights taken from biased
scores, an unstable bucket order) fails at least one of them.
"""
import itertools
import math

import numpy as np
import pytest

import oracle
import synth


# ------------------------------------------------------------------ decode ---

def test_e2m1_table_matches_pages(golden):
    rows = golden("e2m1_values.txt")
    assert len(rows) == 16
    for code, (val,) in rows:
        got = oracle.e2m1(int(code))
        assert got == float(val)
        assert math.copysign(1.0, got) == math.copysign(1.0, float(val)), "sign of zero"


def test_e8m0_all_bytes():
    # 2^(s-127) for every byte (pages: value = E2M1 * 2^(scale-127)); 255 is NaN.
    for s in range(255):
        assert oracle.e8m0(s) == math.ldexp(1.0, s - 127)
    assert math.isnan(oracle.e8m0(255))
    assert oracle.e8m0(127) == 1.0 and oracle.e8m0(121) == 1 / 64 and oracle.e8m0(125) == 0.25


def _blocks(golden):
    rows = golden("mxfp4_hand_blocks.txt")
    blocks, cur = [], None
    for key, vals in rows:
        if key == "block":
            cur = {"name": vals[0]}
            blocks.append(cur)
        elif key == "bytes":
            cur["bytes"] = np.array([int(v, 16) for v in vals], np.uint8)
        elif key == "scale":
            cur["scale"] = int(vals[0])
        elif key == "values":
            cur["values"] = [float(v) for v in vals]
    return blocks


def test_hand_worked_blocks(golden):
    blocks = _blocks(golden)
    assert len(blocks) == 4
    for b in blocks:
        scl = np.array([b["scale"]], np.uint8)
        got = oracle.decode_matrix(b["bytes"], scl, 1, 32)[0]
        assert list(got) == b["values"], b["name"]
        for c in range(32):
            assert oracle.mx_elem(b["bytes"], scl, 32, 0, c) == b["values"][c]


def test_scale_block_and_row_indexing():
    # 2 rows x 64 cols: every (row, 32-block) has its own scale, every byte is code 2 (1.0) in
    # both nibbles, so element (r, c) must equal the scale of (r, c // 32).  A transposed
    # scale index or a per-row-only scale fails.
    nib = np.full(2 * 32, 0x22, np.uint8)
    scl = np.array([121, 122, 123, 124], np.uint8)
    m = oracle.decode_matrix(nib, scl, 2, 64)
    for r in range(2):
        for c in range(64):
            assert m[r, c] == 2.0 ** (int(scl[r * 2 + c // 32]) - 127)
    # distinct nibbles along a row: element c of row 1 is code (c % 16) of the ramp
    ramp = np.array([0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE] * 4, np.uint8)
    nib2 = np.concatenate([np.zeros(32, np.uint8), ramp])
    m2 = oracle.decode_matrix(nib2, np.full(4, 127, np.uint8), 2, 64)
    assert np.all(m2[0] == 0)
    for c in range(64):
        assert m2[1, c] == oracle.e2m1(c % 16)


def test_k3_expert_size(golden):
    g = dict((k, v[0]) for k, v in golden("k3_expert_size.txt"))
    d, f = int(g["d"]), int(g["f"])
    nb, sb = oracle.expert_bytes(d, f)
    assert 3 * d * f == int(g["expert_params"])
    assert nb + sb == int(g["expert_bytes"])
    assert (nb + sb) / (3 * d * f) == float(g["bytes_per_param"])
    fp32 = int(g["experts_per_token"]) * 3 * d * f * 4
    assert round(fp32 / 1e9) == int(g["fp32_expanded_per_token_gb"])
    # the generator's canonical sizes agree with the oracle's
    assert synth.expert_bytes(d, f) == (nb, sb)


# ------------------------------------------------------------------ router ---

def _hand_router_inputs(golden):
    g = dict(golden("router_hand.txt"))
    logits = [float(v) for v in g["logits"]]
    d, E = 32, 4
    x = np.zeros((1, d), np.uint16)
    x[0, 0] = 0x3F80  # bf16 1.0
    Wr = np.zeros((E, d), np.float32)
    Wr[:, 0] = logits
    return g, x, Wr


def test_router_hand_example_bias_selects_only(golden):
    g, x, Wr = _hand_router_inputs(golden)
    bias = np.array([float(v) for v in g["bias"]], np.float32)
    idx, w, logits, keys = oracle.router(x, Wr, bias, 2)
    assert list(idx[0]) == [int(v) for v in g["idx_bias"]]
    np.testing.assert_allclose(w[0], [float(v) for v in g["w_bias"]], rtol=0, atol=1e-15)
    idx0, w0, _, _ = oracle.router(x, Wr, None, 2)
    assert list(idx0[0]) == [int(v) for v in g["idx_nobias"]]
    np.testing.assert_allclose(w0[0], [float(v) for v in g["w_nobias"]], rtol=0, atol=1e-15)


def test_router_logits_against_library_matmul():
    T, d, E = 5, 256, 8
    x = synth.tokens_bf16(7, 0, 0, T, d)
    Wr = synth.router_weights(7, 0, E, d)
    _, _, logits, _ = oracle.router(x, Wr, None, 2)
    ref = synth.bf16_bits_to_f32(x).astype(np.float64) @ Wr.astype(np.float64).T
    np.testing.assert_allclose(logits, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("E,k,T", [(8, 2, 6), (12, 3, 4), (10, 5, 3), (6, 6, 2)])
def test_router_topk_brute_force(E, k, T):
    d = 64
    x = synth.tokens_bf16(11, 0, 0, T, d)
    Wr = synth.router_weights(11, 0, E, d)
    bias = np.zeros(E, np.float32)
    bias[::3] = 0.25
    idx, w, _, keys = oracle.router(x, Wr, bias, k)
    for t in range(T):
        best = max(itertools.combinations(range(E), k), key=lambda s: sum(keys[t, e] for e in s))
        assert sorted(idx[t]) == sorted(best)
        assert all(keys[t, idx[t, i]] >= keys[t, idx[t, i + 1]] for i in range(k - 1))
        assert abs(w[t].sum() - 1.0) < 1e-12
        assert np.all(w[t] > 0)


def test_router_weights_unbiased_and_k_equals_E():
    # k = E: every expert picked, w = sigma / sum(sigma) whatever the bias is.
    T, d, E = 3, 32, 6
    x = synth.tokens_bf16(5, 0, 0, T, d)
    Wr = synth.router_weights(5, 0, E, d)
    bias = np.linspace(-1, 1, E).astype(np.float32)
    idx, w, logits, keys = oracle.router(x, Wr, bias, E)
    sig = keys - bias.astype(np.float64)[None, :]
    for t in range(T):
        np.testing.assert_allclose(w[t], sig[t, idx[t]] / sig[t].sum(), rtol=1e-14)
        np.testing.assert_allclose(sig[t], 1 / (1 + np.exp(-logits[t])), rtol=1e-14)


def test_router_ties_go_to_lower_id():
    T, d, E, k = 2, 32, 8, 3
    x = synth.tokens_bf16(3, 0, 0, T, d)
    Wr = np.zeros((E, d), np.float32)  # every logit 0, every key 0.5
    idx, w, _, _ = oracle.router(x, Wr, None, k)
    assert idx.tolist() == [[0, 1, 2], [0, 1, 2]]
    np.testing.assert_allclose(w, 1.0 / k, rtol=0, atol=1e-15)


def test_topk_gap_helper():
    keys = np.array([[0.9, 0.1, 0.5, 0.7]])
    assert oracle.topk_gap(keys, 2)[0] == pytest.approx(0.2)
    assert np.isinf(oracle.topk_gap(keys, 4)[0])


# --------------------------------------------------------------- bucketing ---

def test_bucket_hand_example(golden):
    g = dict(golden("bucket_hand.txt"))
    idx = np.array([int(v) for v in g["idx"]], np.int32).reshape(3, 2)
    counts, offsets, perm = oracle.bucket(idx, 4)
    assert counts.tolist() == [int(v) for v in g["counts"]]
    assert offsets.tolist() == [int(v) for v in g["offsets"]]
    assert perm.tolist() == [int(v) for v in g["perm"]]


@pytest.mark.parametrize("T,k,E", [(1, 16, 896), (37, 4, 20), (64, 2, 8), (5, 3, 3)])
def test_bucket_invariants(T, k, E):
    rng = np.random.default_rng(T * 1000 + E)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, perm = oracle.bucket(idx, E)
    flat = idx.reshape(-1)
    assert counts.tolist() == np.bincount(flat, minlength=E).tolist()
    assert offsets[0] == 0 and offsets[-1] == T * k
    assert np.all(np.diff(offsets) == counts)
    assert sorted(perm.tolist()) == list(range(T * k))
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg) > 0), "stable: ascending (t, slot)"


# --------------------------------------------------------------------- FFN ---

def _expert_blocks(nib_mats, scl_mats):
    return np.concatenate([m.reshape(-1) for m in nib_mats]), np.concatenate([s.reshape(-1) for s in scl_mats])


def test_ffn_second_formulation_c1():
    # Expand each matrix to fp64 (decode pinned above), then numpy matmuls.
    d, f = 256, 128
    nib, scl = synth.experts(1, 0, 0, 3, d, f)
    x = synth.bf16_bits_to_f32(synth.tokens_bf16(1, 0, 0, 1, d))[0].astype(np.float64)
    mn, ms = f * d // 2, f * d // 32
    for e in range(3):
        Wg = oracle.decode_matrix(nib[e, :mn], scl[e, :ms], f, d)
        Wu = oracle.decode_matrix(nib[e, mn:2 * mn], scl[e, ms:2 * ms], f, d)
        Wd = oracle.decode_matrix(nib[e, 2 * mn:], scl[e, 2 * ms:], d, f)
        g, u = Wg @ x, Wu @ x
        h_ref = g / (1 + np.exp(-g)) * u
        o_ref = Wd @ h_ref
        a_ref = np.abs(Wd) @ np.abs(h_ref)
        h, o, a = oracle.expert_ffn(d, f, nib[e], scl[e], x)
        np.testing.assert_allclose(h, h_ref, rtol=1e-12, atol=1e-12 * np.abs(g).max() * np.abs(u).max())
        assert np.all(np.abs(o - o_ref) <= 1e-12 * a_ref + 1e-12)
        np.testing.assert_allclose(a, a_ref, rtol=1e-12)


def test_ffn_single_nonzero_closed_form():
    d, f = 64, 32
    r0, j0, j1, i0 = 5, 7, 40, 50
    ng = np.zeros((f, d // 2), np.uint8)
    nu = np.zeros((f, d // 2), np.uint8)
    nd = np.zeros((d, f // 2), np.uint8)
    ng[r0, j0 // 2] = 0x2 << (4 * (j0 % 2))      # W_g[r0, j0] = 1.0
    nu[r0, j1 // 2] = 0x4 << (4 * (j1 % 2))      # W_u[r0, j1] = 2.0
    nd[i0, r0 // 2] = 0x9 << (4 * (r0 % 2))      # W_d[i0, r0] = -0.5
    sg = np.full((f, d // 32), 127, np.uint8)
    su = np.full((f, d // 32), 127, np.uint8)
    sd = np.full((d, f // 32), 127, np.uint8)
    nib, scl = _expert_blocks([ng, nu, nd], [sg, su, sd])
    x = np.zeros(d)
    x[j0], x[j1] = 2.0, 3.0
    h, o, a = oracle.expert_ffn(d, f, nib, scl, x)
    silu2 = 2.0 * 0.8807970779778823              # silu(2) = 2 * sigmoid(2), sigmoid(2) by hand
    expect_h = np.zeros(f)
    expect_h[r0] = silu2 * 6.0
    np.testing.assert_allclose(h, expect_h, rtol=1e-15, atol=0)
    expect_o = np.zeros(d)
    expect_o[i0] = -0.5 * silu2 * 6.0
    np.testing.assert_allclose(o, expect_o, rtol=1e-15, atol=0)
    np.testing.assert_allclose(a, np.abs(expect_o), rtol=1e-15, atol=0)


def test_ffn_zero_nibbles_give_zero():
    d, f = 64, 32
    nb, sb = synth.expert_bytes(d, f)
    nib = np.zeros(nb, np.uint8)
    nib[: nb // 3] = 0x88  # gate all -0: still zero
    scl = np.full(sb, 125, np.uint8)
    x = np.linspace(-3, 3, d)
    h, o, a = oracle.expert_ffn(d, f, nib, scl, x)
    assert np.all(h == 0) and np.all(o == 0) and np.all(a == 0)


# ------------------------------------------------------------------- layer ---

def test_layer_c1_against_second_formulation():
    d, f, E, k, T = 256, 128, 8, 2, 4
    nib, scl = synth.experts(1, 0, 0, E, d, f)
    x = synth.tokens_bf16(1, 0, 0, T, d)
    Wr = synth.router_weights(1, 0, E, d)
    out = oracle.layer(x, Wr, None, k, f, nib, scl)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    mn, ms = f * d // 2, f * d // 32
    mats = []
    for e in range(E):
        mats.append((oracle.decode_matrix(nib[e, :mn], scl[e, :ms], f, d),
                     oracle.decode_matrix(nib[e, mn:2 * mn], scl[e, ms:2 * ms], f, d),
                     oracle.decode_matrix(nib[e, 2 * mn:], scl[e, 2 * ms:], d, f)))
    y_ref = np.zeros((T, d))
    for t in range(T):
        for s in range(k):
            Wg, Wu, Wd = mats[out["idx"][t, s]]
            g, u = Wg @ xf[t], Wu @ xf[t]
            y_ref[t] += out["w"][t, s] * (Wd @ (g / (1 + np.exp(-g)) * u))
    assert np.all(np.abs(out["y"] - y_ref) <= 1e-12 * out["sumabs"] + 1e-12)
    assert np.all(out["sumabs"] >= np.abs(out["y"]) * (1 - 1e-12))


def test_layer_k1_combine_is_identity():
    # k = 1: the single weight is 1, so y equals the chosen expert's o exactly.
    d, f, E = 64, 32, 4
    nib, scl = synth.experts(2, 0, 0, E, d, f)
    x = synth.tokens_bf16(2, 0, 0, 3, d)
    Wr = synth.router_weights(2, 0, E, d)
    out = oracle.layer(x, Wr, None, 1, f, nib, scl)
    assert np.all(out["w"] == 1.0)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    for t in range(3):
        _, o, _ = oracle.expert_ffn(d, f, nib[out["idx"][t, 0]], scl[out["idx"][t, 0]], xf[t])
        assert np.array_equal(out["y"][t], o)


# ------------------------------------------------------ glue between layers ---

def _torch_bf16_bits(v: np.ndarray) -> np.ndarray:
    torch = pytest.importorskip("torch")
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_bf16_rne_hand_values():
    # ulp(1) in bf16 is 2^-7: 1 + 2^-8 is a tie (stays at the even code 1.0), 1 + 3*2^-8 is a
    # tie between 1 + 2^-7 (odd) and 1 + 2^-6 (even), a hair above a tie rounds up.
    assert oracle.bf16_rne(1.0) == 0x3F80
    assert oracle.bf16_rne(1.0 + 2 ** -8) == 0x3F80
    assert oracle.bf16_rne(1.0 + 3 * 2 ** -8) == 0x3F82
    assert oracle.bf16_rne(1.0 + 2 ** -8 + 2 ** -20) == 0x3F81
    assert oracle.bf16_rne(-1.5) == 0xBFC0
    assert oracle.bf16_rne(float("inf")) == 0x7F80
    assert oracle.bf16_rne(3.4e38) == 0x7F80  # above the largest finite bf16: rounds to inf


def test_bf16_rne_matches_library_conversion():
    # a second formulation: torch's float32 -> bfloat16 conversion (round to nearest even)
    rng = np.random.default_rng(3)
    with np.errstate(over="ignore", invalid="ignore"):
        wide = (rng.standard_normal(4000) * 10.0 ** rng.integers(-30, 30, 4000)).astype(np.float32)
    bits = rng.integers(0, 2 ** 32, 4000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    v = np.concatenate([wide, bits])
    v = v[np.isfinite(v)]
    ref = _torch_bf16_bits(v)
    got = np.array([oracle.bf16_rne(float(a)) for a in v], np.uint16)
    assert np.array_equal(got, ref)


def test_residual_is_bf16_of_the_fp32_sum():
    rng = np.random.default_rng(4)
    T, d = 3, 96
    x = synth.tokens_bf16(4, 0, 0, T, d)
    y = (rng.standard_normal((T, d)) * 50).astype(np.float32)
    x_next, _ = oracle.residual_rmsnorm(y, x, 1e-6)
    ref = _torch_bf16_bits(synth.bf16_bits_to_f32(x) + y)
    assert np.array_equal(x_next, ref)


def test_rmsnorm_closed_forms():
    d = 4
    x = np.zeros((2, d), np.uint16)
    # (3, 4, 0, 0): mean square 25/4, root 2.5 -> (1.2, 1.6, 0, 0); constant -7 -> all -1
    y = np.array([[3, 4, 0, 0], [-7, -7, -7, -7]], np.float32)
    _, xn = oracle.residual_rmsnorm(y, x, 0.0)
    assert np.array_equal(xn[0], _torch_bf16_bits(np.array([1.2, 1.6, 0, 0], np.float32)))
    assert np.array_equal(xn[1], np.full(d, 0xBF80, np.uint16))
    # eps enters under the root: (1,1,1,1) with eps = 3 -> 1/2
    _, xn = oracle.residual_rmsnorm(np.ones((1, d), np.float32), np.zeros((1, d), np.uint16), 3.0)
    assert np.array_equal(xn[0], np.full(d, 0x3F00, np.uint16))


def test_rmsnorm_scale_invariance_and_unit_rms():
    rng = np.random.default_rng(5)
    d = 512
    y = rng.standard_normal((1, d)).astype(np.float32)
    z = np.zeros((1, d), np.uint16)
    _, a = oracle.residual_rmsnorm(y, z, 0.0)
    _, b = oracle.residual_rmsnorm(y * np.float32(2.0 ** 40), z, 0.0)
    assert np.array_equal(a, b)
    v = synth.bf16_bits_to_f32(a).astype(np.float64)
    assert abs(np.mean(v * v) - 1.0) < 2 * 2 ** -8


# ------------------------------------------------------------------ SiTU-GLU ---
# The deep dive's glossary entry SiTU-GLU gives K3's activation only as a tanh-sigmoid
# combination whose beta1 = 4 and beta2 = 25 bound the gate above by 100.  The formula is a
# reading (parity unpinned); these pins tie the oracle to what the page fixes (the bound 100)
# and to the limits and slope that the reading implies, and check where the gate sits in the FFN.

def test_situ_bound_is_beta1_times_beta2():
    assert oracle.situ(1000.0) == pytest.approx(100.0, rel=1e-15)   # beta1 * beta2, from the page
    zs = np.linspace(-300.0, 300.0, 6001)
    vals = np.array([oracle.situ(z) for z in zs])
    assert vals.max() <= 100.0 and oracle.situ(200.0) > 99.9999


def test_situ_limits_and_slope():
    assert oracle.situ(0.0) == 0.0
    assert abs(oracle.situ(-1000.0)) < 1e-300                        # sigmoid -> 0
    eps = 1e-6
    slope = (oracle.situ(eps) - oracle.situ(-eps)) / (2 * eps)
    assert slope == pytest.approx(4.0 / 2.0, rel=1e-9)               # beta1 * beta2 * (1/2) * (1/beta2)
    # for large positive gates the sigmoid is 1 and the gate is the capped tanh: 100 tanh(z / 25)
    assert oracle.situ(50.0) == pytest.approx(100.0 * np.tanh(2.0), rel=1e-15)


def test_ffn_situ_gate_applies_to_g_not_u():
    # single nonzero weights (the closed-form case above): h = situ(g) * u with g = 2, u = 6
    d, f = 64, 32
    r0, j0, j1, i0 = 5, 7, 40, 50
    ng = np.zeros((f, d // 2), np.uint8)
    nu = np.zeros((f, d // 2), np.uint8)
    nd = np.zeros((d, f // 2), np.uint8)
    ng[r0, j0 // 2] = 0x2 << (4 * (j0 % 2))      # W_g[r0, j0] = 1.0
    nu[r0, j1 // 2] = 0x4 << (4 * (j1 % 2))      # W_u[r0, j1] = 2.0
    nd[i0, r0 // 2] = 0x9 << (4 * (r0 % 2))      # W_d[i0, r0] = -0.5
    sg = np.full((f, d // 32), 127, np.uint8)
    su = np.full((f, d // 32), 127, np.uint8)
    sd = np.full((d, f // 32), 127, np.uint8)
    nib, scl = _expert_blocks([ng, nu, nd], [sg, su, sd])
    x = np.zeros(d)
    x[j0], x[j1] = 2.0, 3.0
    h, o, _ = oracle.expert_ffn(d, f, nib, scl, x, act=oracle.ACT_SITU_GLU)
    assert h[r0] == pytest.approx(oracle.situ(2.0) * 6.0, rel=1e-15)
    assert np.count_nonzero(h) == 1
    assert o[i0] == pytest.approx(-0.5 * oracle.situ(2.0) * 6.0, rel=1e-15)


def test_ffn_situ_second_formulation():
    d, f = 256, 128
    nib, scl = synth.experts(2, 0, 0, 2, d, f)
    x = synth.bf16_bits_to_f32(synth.tokens_bf16(2, 0, 0, 1, d))[0].astype(np.float64)
    mn, ms = f * d // 2, f * d // 32
    situ = np.vectorize(oracle.situ)
    for e in range(2):
        Wg = oracle.decode_matrix(nib[e, :mn], scl[e, :ms], f, d)
        Wu = oracle.decode_matrix(nib[e, mn:2 * mn], scl[e, ms:2 * ms], f, d)
        Wd = oracle.decode_matrix(nib[e, 2 * mn:], scl[e, 2 * ms:], d, f)
        h_ref = situ(Wg @ x) * (Wu @ x)
        o_ref = Wd @ h_ref
        h, o, a = oracle.expert_ffn(d, f, nib[e], scl[e], x, act=oracle.ACT_SITU_GLU)
        np.testing.assert_allclose(h, h_ref, rtol=1e-12, atol=1e-12 * np.abs(h_ref).max())
        assert np.all(np.abs(o - o_ref) <= 1e-12 * (np.abs(Wd) @ np.abs(h_ref)) + 1e-12)
