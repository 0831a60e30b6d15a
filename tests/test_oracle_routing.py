"""Pins of the oracle's router logits, top-k, weights and permutation."""
import json
import os

import numpy as np
import pytest

import oracle
from conftest import GOLDEN


def _bf16(a):
    return oracle.f32_to_bf16(np.asarray(a, np.float32))


def test_logit_summation_order_fixed():
    # x = 1 everywhere; w[0] = 2^24, w[128] = -2^24, all other w = 1.
    # In the fixed order lane 0 holds elements 0..7 and lane 16 holds 128..135:
    # lane 0 = 2^24 (each +1 rounds back to 2^24), lane 16 = -2^24 + 7 (exact),
    # the 30 other lanes = 8.  Level d=16: lane 0 = 7, lanes 1..15 = 16;
    # d=8: 7 + 16 = 23; d=4: 23 + 32 = 55; d=2: 55 + 64 = 119; d=1: 119 + 128 = 247.
    # (A left-to-right fp32 sum would give 127, the exact sum is 254.)
    H = 256
    x = _bf16(np.ones((1, H)))
    w = np.ones((1, H), np.float32)
    w[0, 0] = 2.0 ** 24
    w[0, 128] = -(2.0 ** 24)
    lg = oracle.router_logits(x, _bf16(w), None)
    assert lg[0, 0] == np.float32(247.0)
    lg = oracle.router_logits(x, _bf16(w), np.array([0.5], np.float32))
    assert lg[0, 0] == np.float32(247.5)


def test_logits_close_to_exact_dot():
    rng = np.random.default_rng(11)
    T, H, E = 5, 1024, 40
    x = _bf16(rng.standard_normal((T, H)))
    wr = _bf16(rng.standard_normal((E, H)) * 0.05)
    bias = rng.standard_normal(E).astype(np.float32)
    lg = oracle.router_logits(x, wr, bias)
    xf, wf = oracle.bf16_to_f32(x).astype(np.float64), oracle.bf16_to_f32(wr).astype(np.float64)
    exact = xf @ wf.T + bias.astype(np.float64)
    absdot = np.abs(xf) @ np.abs(wf).T
    bound = (H / 32 + 6) * 2.0 ** -24 * absdot + 2.0 ** -24 * np.abs(exact)
    assert np.all(np.abs(lg - exact) <= bound)


def test_onehot_logit_is_the_weight():
    H, E = 256, 3
    x = np.zeros((1, H), np.float32)
    x[0, 77] = 1.0
    wr = np.random.default_rng(1).standard_normal((E, H)).astype(np.float32)
    lg = oracle.router_logits(_bf16(x), _bf16(wr), None)
    np.testing.assert_array_equal(lg[0], oracle.bf16_to_f32(_bf16(wr))[:, 77])


def test_topk_matches_exhaustive_sort_with_ties():
    rng = np.random.default_rng(5)
    T, E, k = 64, 48, 6
    lg = rng.integers(-5, 5, size=(T, E)).astype(np.float32)   # many exact ties
    lg[0, :] = 0.0
    lg[0, 10] = -0.0                                           # -0 ties +0
    idx, w = oracle.topk(lg, k)
    for t in range(T):
        order = np.lexsort((np.arange(E), -lg[t].astype(np.float64)))  # logit desc, index asc
        assert list(idx[t]) == list(order[:k])
    assert list(idx[0]) == [0, 1, 2, 3, 4, 5]


def test_topk_weights_closed_forms():
    lg = np.array([[3.0, 1.0, -2.0, 0.5]], np.float32)
    idx, w = oracle.topk(lg, 2)
    assert list(idx[0]) == [0, 1]
    assert w[0, 0] == pytest.approx(1.0 / (1.0 + np.exp(-2.0)), rel=1e-15)
    idx, w = oracle.topk(lg, 1)
    assert w[0, 0] == 1.0
    eq = np.zeros((1, 8), np.float32)
    idx, w = oracle.topk(eq, 4)
    np.testing.assert_allclose(w[0], 0.25, rtol=1e-15)
    rng = np.random.default_rng(2)
    idx, w = oracle.topk(rng.standard_normal((50, 30)).astype(np.float32) * 4, 5)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-12)
    assert np.all(np.diff(w, axis=1) <= 0)


def test_permutation_invariants():
    rng = np.random.default_rng(9)
    T, E, k = 37, 20, 4
    lg = rng.standard_normal((T, E)).astype(np.float32)
    idx, _ = oracle.topk(lg, k)
    counts, offsets, perm, inv = oracle.permute(idx, E)
    assert counts.sum() == T * k and offsets[0] == 0 and offsets[-1] == T * k
    assert np.all(np.diff(offsets) == counts)
    assert sorted(perm) == list(range(T * k))
    assert np.all(inv[perm] == np.arange(T * k))
    # (expert asc, token asc) order and each token exactly k times with k distinct experts
    ex = idx.ravel()[perm]
    tok = perm // k
    keys = ex.astype(np.int64) * T + tok
    assert np.all(np.diff(keys) > 0)
    for t in range(T):
        assert np.sum(tok == t) == k and len(set(idx[t])) == k


def test_hand_example_routing():
    g = json.load(open(os.path.join(GOLDEN, "hand_example_2experts.json")))
    lg = np.array(g["logits"], np.float32)
    idx, w = oracle.topk(lg, 2)
    assert idx.tolist() == g["k2"]["idx"]
    np.testing.assert_allclose(w, g["k2"]["w"], rtol=1e-8)
    counts, offsets, perm, inv = oracle.permute(idx, 2)
    assert counts.tolist() == g["k2"]["counts"]
    assert offsets.tolist() == g["k2"]["offsets"]
    assert perm.tolist() == g["k2"]["perm"]
