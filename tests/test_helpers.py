"""The parity helpers themselves (CPU): the top-k validity check used for near-tie tokens accepts
the oracle's own routing and rejects a wrong set, a wrong slot order and wrong weights."""
import numpy as np
import pytest

import oracle
import synth
from helpers import assert_routing_valid


def _routing(T=6, d=64, E=12, k=3):
    x = synth.tokens_bf16(31, 0, 0, T, d)
    Wr = synth.router_weights(31, 0, E, d)
    idx, w, logits, keys = oracle.router(x, Wr, None, k)
    return idx, w.astype(np.float32), logits, keys


def test_accepts_the_oracle_routing():
    idx, w, logits, keys = _routing()
    assert_routing_valid(idx, w, logits, keys, 1e-9)


def test_rejects_a_set_that_is_not_a_top_k():
    idx, w, logits, keys = _routing()
    bad = idx.copy()
    order = np.argsort(-keys[0])
    bad[0, -1] = order[-1]  # the smallest key instead of the k-th largest
    with pytest.raises(AssertionError, match="top-3"):
        assert_routing_valid(bad, w, logits, keys, 1e-9)


def test_rejects_slots_out_of_key_order():
    idx, w, logits, keys = _routing()
    gaps = keys[np.arange(len(idx))[:, None], idx]
    t = int(np.argmax(gaps[:, 0] - gaps[:, 1]))  # a token whose first two keys are well apart
    bad, wb = idx.copy(), w.copy()
    bad[t, [0, 1]] = bad[t, [1, 0]]
    wb[t, [0, 1]] = wb[t, [1, 0]]
    with pytest.raises(AssertionError, match="key order"):
        assert_routing_valid(bad, wb, logits, keys, 1e-9)


def test_rejects_wrong_weights_and_repeated_picks():
    idx, w, logits, keys = _routing()
    wb = w.copy()
    wb[2, 0] += 1e-3
    with pytest.raises(AssertionError, match="weights"):
        assert_routing_valid(idx, wb, logits, keys, 1e-9)
    bad = idx.copy()
    bad[1, 1] = bad[1, 0]
    with pytest.raises(AssertionError, match="bad picks"):
        assert_routing_valid(bad, w, logits, keys, 1e-9)
