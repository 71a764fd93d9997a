"""Pins of the oracle router (softmax over E, top-k, renormalise over k)."""

import itertools
import math

import numpy as np

from moe_inputs import synth, bf16_bits_to_f64
from oracle.routing import router_logits, softmax, topk_ascending, route


def _tiny_route():
    s = synth(1)
    wl = s.wl
    x = bf16_bits_to_f64(s.tokens(0, 0))
    _, wr, b = s.router(0)
    return wl, x, wr, b


def test_brute_force_subset_on_tiny_layer():
    # the chosen set is the k-subset of experts with the largest summed logit
    wl, x, wr, b = _tiny_route()
    idx, w, l = route(x, wr, b, wl.top_k)
    for t in range(x.shape[0]):
        best = max(itertools.combinations(range(wl.n_experts), wl.top_k),
                   key=lambda c: sum(l[t, e] for e in c))
        assert tuple(idx[t]) == best


def test_brute_force_probability_product():
    # equivalently the subset with the largest product of softmax probabilities
    rng = np.random.default_rng(11)
    l = rng.standard_normal((6, 9))
    p = softmax(l)
    got = topk_ascending(l, 3)
    for t in range(6):
        best = max(itertools.combinations(range(9), 3), key=lambda c: math.prod(p[t, e] for e in c))
        assert tuple(got[t]) == best


def test_ties_go_to_lower_id():
    l = np.array([[1.0, 2.0, 2.0, 0.5, 2.0]])
    assert topk_ascending(l, 2).tolist() == [[1, 2]]
    assert topk_ascending(l, 3).tolist() == [[1, 2, 4]]
    assert topk_ascending(np.zeros((1, 5)), 2).tolist() == [[0, 1]]


def test_renormalised_weights_equal_softmax_over_chosen_logits():
    wl, x, wr, b = _tiny_route()
    idx, w, l = route(x, wr, b, wl.top_k)
    for t in range(x.shape[0]):
        lc = l[t, idx[t]]
        closed = np.exp(lc - lc.max()) / np.exp(lc - lc.max()).sum()
        assert np.allclose(w[t], closed, rtol=0, atol=1e-14)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-12)
    for t in range(x.shape[0]):
        assert len(set(idx[t].tolist())) == wl.top_k
        assert np.all(np.diff(idx[t]) > 0)


def test_softmax_closed_form_and_shift_invariance():
    p = softmax(np.array([[0.0, math.log(2.0), math.log(3.0)]]))
    assert np.allclose(p, [[1 / 6, 2 / 6, 3 / 6]], atol=1e-15)
    rng = np.random.default_rng(4)
    l = rng.standard_normal((3, 50)) * 30
    assert np.allclose(softmax(l), softmax(l + 123.0), atol=1e-15)
    assert np.all(np.isfinite(softmax(l * 100)))


def test_one_hot_input_selects_router_column():
    s = synth(2)
    _, wr, b = s.router(0)
    for j in (0, 777, 2047):
        x = np.zeros((1, 2048))
        x[0, j] = 1.0
        assert np.array_equal(router_logits(x, wr, b)[0], wr[:, j])


def test_full_size_route_counts():
    # 10 distinct routed experts per token, weights sum to 1 (page 1, §如何做到：三层存储)
    s = synth(2)
    x = bf16_bits_to_f64(s.tokens_many(0, list(range(8))).reshape(-1, 2048))
    _, wr, b = s.router(0)
    idx, w, _ = route(x, wr, b, 10)
    assert idx.shape == (8, 10)
    assert all(len(set(r)) == 10 for r in idx.tolist())
    assert np.allclose(w.sum(1), 1, atol=1e-12) and np.all(w > 0)


def test_one_hot_input_with_bias_adds_bias():
    s = synth(3)
    _, wr, b = s.router(7)
    assert np.any(b != 0)
    x = np.zeros((2, 2048))
    x[0, 5] = 1.0
    x[1, 5] = -2.0
    l = router_logits(x, wr, b)
    assert np.array_equal(l[0], wr[:, 5] + b.astype(np.float64))
    assert np.array_equal(l[1], -2.0 * wr[:, 5] + b.astype(np.float64))
    # with a dominant bias the chosen set is the k lowest Zipf ranks
    idx, w, _ = route(np.zeros((1, 2048)), wr, b * 100, 10)
    ranks = np.rint(np.exp(-b.astype(np.float64) / (s.bias_lambda * 1.1))).astype(int)
    assert sorted(ranks[idx[0]].tolist()) == list(range(1, 11))
