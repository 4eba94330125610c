"""Shared test helpers: seeded workloads, the gap filter, and the parity comparisons."""
from __future__ import annotations

import numpy as np

import oracle
import synth

GAP_MIN = 1e-3      # oracle key gap between the k-th and (k+1)-th expert, per token
ORDER_GAP = 1e-5    # slot order is compared where adjacent oracle keys differ by more than this
REL_TOL = 2e-3      # |y_gpu - y_oracle| <= REL_TOL * sum|terms| + ABS_TOL
ABS_TOL = 1e-5


def gap_filtered_tokens(seed, layer, t0, T, d, Wr, bias, k, max_attempts=64):
    """Tokens t0..t0+T-1, each redrawn (attempt += 1) until the oracle's k-th/(k+1)-th key gap
    is at least GAP_MIN.  Returns (x_bits uint16[T,d], attempts int32[T])."""
    attempts = np.zeros(T, np.int32)
    x = synth.tokens_bf16(seed, layer, t0, T, d, attempts)
    if k >= Wr.shape[0]:
        return x, attempts
    todo = np.arange(T)
    for _ in range(max_attempts):
        _, _, _, keys = oracle.router(x[todo], Wr, bias, k)
        bad = todo[oracle.topk_gap(keys, k) < GAP_MIN]
        if bad.size == 0:
            return x, attempts
        attempts[bad] += 1
        for t in bad:
            x[t] = synth.tokens_bf16(seed, layer, t0 + int(t), 1, d, attempts[t:t + 1])[0]
        todo = bad
    raise RuntimeError("gap filter did not converge")


def assert_routing_matches(idx_gpu, w_gpu, idx_o, w_o, keys_o):
    """Top-k sets exactly equal; slot order equal wherever the oracle keys are separated;
    combine weights within fp32 rounding (matched by expert id)."""
    T, k = idx_o.shape
    for t in range(T):
        assert sorted(idx_gpu[t].tolist()) == sorted(idx_o[t].tolist()), f"token {t}: top-k set differs"
        ko = keys_o[t, idx_o[t]]
        for i in range(k):
            sep_prev = i == 0 or ko[i - 1] - ko[i] > ORDER_GAP
            sep_next = i == k - 1 or ko[i] - ko[i + 1] > ORDER_GAP
            if sep_prev and sep_next:
                assert idx_gpu[t, i] == idx_o[t, i], f"token {t}: slot {i} order differs"
        wg = dict(zip(idx_gpu[t].tolist(), w_gpu[t].tolist()))
        for e, wo in zip(idx_o[t].tolist(), w_o[t].tolist()):
            assert abs(wg[e] - wo) <= 1e-5 * max(1.0, abs(wo)), f"token {t}: weight of expert {e}"


def assert_routing_valid(idx_gpu, w_gpu, logits_o, keys_o, tol):
    """For tokens whose k-th and (k+1)-th oracle keys may be closer than the GPU's rounding: the
    GPU's picks are k distinct experts that form a top-k of the oracle keys within `tol` (no
    unpicked key above a picked one by more than tol), in descending key order within tol, and
    the weights are the oracle's sigmoid scores of the GPU's own picks, renormalised (within
    1e-5)."""
    T, k = idx_gpu.shape
    E = keys_o.shape[1]
    sig = 1.0 / (1.0 + np.exp(-logits_o))
    for t in range(T):
        pick = idx_gpu[t].astype(np.int64)
        assert len(set(pick.tolist())) == k and pick.min() >= 0 and pick.max() < E, f"token {t}: bad picks"
        rest = np.setdiff1d(np.arange(E), pick)
        kp = keys_o[t, pick]
        if rest.size:
            assert kp.min() >= keys_o[t, rest].max() - tol, f"token {t}: not a top-{k} within {tol}"
        assert (np.diff(kp) <= tol).all(), f"token {t}: slots out of key order"
        wo = sig[t, pick] / sig[t, pick].sum()
        assert np.abs(w_gpu[t] - wo).max() <= 1e-5, f"token {t}: weights"


def assert_y_close(y_gpu, y_o, sumabs, what=""):
    err = np.abs(y_gpu.astype(np.float64) - y_o)
    bound = REL_TOL * sumabs + ABS_TOL
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside bound; first at {tuple(i)}: "
                             f"gpu {y_gpu[tuple(i)]} oracle {y_o[tuple(i)]} bound {bound[tuple(i)]}")
    return float((err / np.maximum(sumabs, 1e-30)).max())


def unpack_tiles(packed: np.ndarray, d: int, f: int):
    """Invert the packed tile layout (the spec in k3moe_internal.cuh, restated independently here)
    back to canonical (nib, scl) for one expert."""
    TB = 1088
    out_nib = []
    out_scl = []
    gu_tiles = (f // 16) * (d // 128) * 2
    for m, (R, K) in enumerate([(f, d), (f, d), (d, f)]):
        nib = np.zeros((R, K // 2), np.uint8)
        scl = np.zeros((R, K // 32), np.uint8)
        for rg in range(R // 16):
            for kt in range(K // 128):
                if m < 2:
                    tile = ((rg * (d // 128) + kt) * 2 + m)
                else:
                    tile = gu_tiles + rg * (f // 128) + kt
                tb = packed[tile * TB:(tile + 1) * TB]
                for u in range(2):
                    for lane in range(32):
                        g, t = lane // 4, lane % 4
                        for s in range(4):
                            kb = kt * 128 + 64 * u + 16 * s
                            w = tb[u * 512 + lane * 16 + 4 * s: u * 512 + lane * 16 + 4 * s + 4]
                            nib[rg * 16 + g, (kb + 2 * t) // 2] = w[0]
                            nib[rg * 16 + g + 8, (kb + 2 * t) // 2] = w[1]
                            nib[rg * 16 + g, (kb + 2 * t + 8) // 2] = w[2]
                            nib[rg * 16 + g + 8, (kb + 2 * t + 8) // 2] = w[3]
                for g in range(8):
                    for h in range(2):
                        for b in range(4):
                            scl[rg * 16 + g + 8 * h, kt * 4 + b] = tb[1024 + 8 * g + 4 * h + b]
        out_nib.append(nib.reshape(-1))
        out_scl.append(scl.reshape(-1))
    return np.concatenate(out_nib), np.concatenate(out_scl)
