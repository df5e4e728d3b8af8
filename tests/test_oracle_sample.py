"""Pins of the oracle's sampling decoding (top-k / top-p restriction, inverse CDF at a given
uniform u), CPU only: closed forms on hand-made probabilities, the exact frequencies of a
uniform grid of u, greedy limits, invariances, and the log-probability against scipy."""
import numpy as np
import pytest
from scipy.special import logsumexp, softmax

import oracle


def _grid(n):
    return (np.arange(n) + 0.5) / n


def test_top_k_one_is_greedy():
    g = np.random.default_rng(0)
    x = g.standard_normal((20, 300)).astype(np.float32)
    r = oracle.sample(x, g.random(20), top_k=1)
    np.testing.assert_array_equal(r["token"], x.argmax(axis=1))


def test_uniform_grid_hits_the_renormalised_top_k_probabilities():
    # probabilities 0.4, 0.3, 0.2, 0.1 on tokens 7, 2, 9, 4; the rest far below
    p = {7: 0.4, 2: 0.3, 9: 0.2, 4: 0.1}
    x = np.full(12, -40.0, np.float32)
    for v, pv in p.items():
        x[v] = np.log(pv)
    n = 1000
    for top_k, kept in ((4, [7, 2, 9, 4]), (3, [7, 2, 9]), (2, [7, 2])):
        r = oracle.sample(np.tile(x, (n, 1)), _grid(n), top_k=top_k)
        tot = sum(p[v] for v in kept)
        counts = {v: int((r["token"] == v).sum()) for v in kept}
        for v in kept:
            assert abs(counts[v] - n * p[v] / tot) <= 1, (top_k, counts)
        assert sum(counts.values()) == n


def test_top_p_keeps_the_shortest_prefix_reaching_p():
    p = [0.5, 0.3, 0.2]
    x = np.log(np.array(p)).astype(np.float32)
    n = 800
    # top_p 0.75: 0.5 < 0.75 <= 0.8  ->  tokens 0, 1 renormalised to 0.625 / 0.375
    r = oracle.sample(np.tile(x, (n, 1)), _grid(n), top_k=3, top_p=0.75)
    assert abs((r["token"] == 0).sum() - 0.625 * n) <= 1 and (r["token"] == 2).sum() == 0
    # top_p 0.5 is reached by the first token alone
    r = oracle.sample(np.tile(x, (n, 1)), _grid(n), top_k=3, top_p=0.5)
    assert (r["token"] == 0).all()
    # top_p 1 changes nothing
    a = oracle.sample(np.tile(x, (n, 1)), _grid(n), top_k=3, top_p=1.0)
    b = oracle.sample(np.tile(x, (n, 1)), _grid(n), top_k=3)
    np.testing.assert_array_equal(a["token"], b["token"])


def test_extreme_u_picks_the_ends_of_the_kept_set():
    g = np.random.default_rng(2)
    x = g.standard_normal((30, 500)).astype(np.float32)
    order = np.argsort(-x, axis=1, kind="stable")
    lo = oracle.sample(x, np.zeros(30), top_k=8)
    hi = oracle.sample(x, np.full(30, 1 - 1e-12), top_k=8)
    np.testing.assert_array_equal(lo["token"], order[:, 0])
    np.testing.assert_array_equal(hi["token"], order[:, 7])


def test_ties_take_the_smaller_token_first():
    x = np.zeros((1, 10), np.float32)
    r = oracle.sample(np.tile(x, (100, 1)), _grid(100), top_k=3)
    assert set(r["token"].tolist()) == {0, 1, 2}


def test_logprob_and_invariances():
    g = np.random.default_rng(3)
    x = (g.standard_normal((16, 1000)) * 2).astype(np.float32)
    u = g.random(16)
    r = oracle.sample(x, u, top_k=5, top_p=0.9)
    want = x.astype(np.float64)[np.arange(16), r["token"]] - logsumexp(x.astype(np.float64), axis=1)
    np.testing.assert_allclose(r["logprob"], want, rtol=0, atol=1e-12)
    # a constant per row changes nothing; a permutation of the vocab permutes the token
    s = oracle.sample(x + np.float32(3.0), u, top_k=5, top_p=0.9)
    np.testing.assert_array_equal(s["token"], r["token"])
    perm = g.permutation(1000)
    inv = np.argsort(perm)
    t = oracle.sample(x[:, perm], u, top_k=5, top_p=0.9)
    np.testing.assert_array_equal(perm[t["token"]], r["token"])


def test_sampling_frequencies_match_softmax_over_top_k():
    g = np.random.default_rng(4)
    x = g.standard_normal(50).astype(np.float32)
    n = 4000
    r = oracle.sample(np.tile(x, (n, 1)), _grid(n), top_k=6)
    top = np.argsort(-x, kind="stable")[:6]
    p = softmax(x[top].astype(np.float64))
    for v, pv in zip(top, p):
        assert abs((r["token"] == v).sum() - n * pv) <= 1


def test_bad_arguments_are_rejected():
    with pytest.raises(ValueError):
        oracle.sample(np.zeros((1, 4), np.float32), [0.5], top_k=5)
    with pytest.raises(ValueError):
        oracle.sample(np.zeros((1, 4), np.float32), [0.5], top_k=2, top_p=0.0)


def test_margin_is_the_distance_to_the_nearest_boundary():
    """The margin the GPU comparison excuses by: the distance of u from the nearest cumulative
    boundary of the kept set (and of top_p from one of the top_k's), on hand-made probabilities
    whose normalised cumulative sums are known: 0.5, 0.8, 1.0."""
    x = np.log(np.array([0.5, 0.3, 0.2, 1e-30], np.float64)).astype(np.float32)
    rows = np.tile(x, (6, 1))
    u = np.array([0.45, 0.79, 0.62, 0.1, 0.999, 0.5001])
    r = oracle.sample(rows, u, top_k=3)
    # kept boundaries at 0.5 and 0.8 (the last, 1.0, is not a boundary)
    want = [0.05, 0.01, 0.12, 0.4, 0.199, 0.0001]
    np.testing.assert_allclose(r["margin"], want, rtol=0, atol=1e-6)
    np.testing.assert_array_equal(r["token"], [0, 1, 1, 0, 2, 1])
    # top_p 0.75 keeps tokens 0, 1 (cumulative 0.625 inside the kept set); the cut's own
    # margin is min |{0.5, 0.8, 1.0} - 0.75| = 0.05
    r = oracle.sample(rows[:3], np.array([0.6, 0.1, 0.64]), top_k=3, top_p=0.75)
    np.testing.assert_allclose(r["margin"], [0.025, 0.05, 0.015], rtol=0, atol=1e-6)
    # a single kept candidate has no boundary: the margin is its ceiling, 1
    r = oracle.sample(rows[:2], np.array([0.3, 0.9]), top_k=1)
    np.testing.assert_array_equal(r["margin"], [1.0, 1.0])
    # a planted mistake a margin of 0 everywhere would excuse every row: the pins above fail it
    assert (oracle.sample(rows, u, top_k=3)["margin"] > 0).all()
