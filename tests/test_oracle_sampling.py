"""Pins for the sampling oracle (``oracle/sampling.py``): the page's worked top-2
example, greedy ties, closed forms for temperature and top-p, and exact frequencies of
the inverse-CDF draw over a grid of uniforms.  Each pin is a ``check_*`` function of the
module under test, so that the mutation test can run them against planted mistakes."""
import math
import os

import numpy as np
import pytest

from oracle import sampling as _sampling

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "sampling_top2_example.txt")


def _example():
    rows = [l.split() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    names = [r[0] for r in rows]
    p = np.array([float(r[1]) for r in rows])
    p2 = np.array([float(r[2]) for r in rows])
    return names, p, p2


def check_top2_example_of_the_page(sampling):
    # logits = log p reproduce the page's distribution at temperature 1
    names, p, p2 = _example()
    logits = np.log(p).astype(np.float32)
    order, w = sampling.candidates(logits, 1.0, 2, 1.0)
    assert [names[i] for i in order] == ["mat", "floor"]
    probs = np.array(w) / sum(w)
    assert np.allclose(probs, p2[:2], atol=1e-6)
    # table and car are never drawn; u below 0.6 gives mat, above gives floor
    for u in np.linspace(0, 0.999, 200):
        got = names[sampling.sample(logits, 1.0, 2, 1.0, float(u))]
        assert got == ("mat" if u < 0.6 - 1e-6 else "floor") or abs(u - 0.6) < 1e-6


def check_greedy_is_the_first_largest(sampling):
    x = np.array([0.5, 2.0, -1.0, 2.0, 1.9], dtype=np.float32)
    for u in (0.0, 0.5, 0.999):
        assert sampling.sample(x, 0.0, 0, 1.0, u) == 1
        assert sampling.sample(x, 0.0, 3, 0.5, u) == 1
    # top-k of 1 is greedy whatever the temperature or u
    for u in (0.0, 0.3, 0.999):
        assert sampling.sample(x, 2.5, 1, 1.0, u) == 1


def check_top_k_order_breaks_ties_by_lower_index(sampling):
    x = np.array([1.0, 3.0, 3.0, 0.0, 3.0], dtype=np.float32)
    order, _ = sampling.candidates(x, 1.0, 4, 1.0)
    assert order == [1, 2, 4, 0]


def check_temperature_is_a_power_of_the_distribution(sampling):
    # softmax(l / T) = p^(1/T) / sum p^(1/T) for l = log p (closed form)
    _, p, _ = _example()
    logits = np.log(p).astype(np.float32)
    for T in (0.7, 1.0, 1.5):
        order, w = sampling.candidates(logits, T, 0, 1.0)
        assert order == [0, 1, 2, 3]
        want = p ** (1.0 / T) / np.sum(p ** (1.0 / T))
        assert np.allclose(np.array(w) / sum(w), want, atol=1e-6)
    # sharper below 1, flatter above (the page's direction; its printed numbers are
    # illustrations: the formula gives mat 0.530 at T = 0.7, not 0.60)
    w07 = np.array(sampling.candidates(logits, 0.7, 0, 1.0)[1])
    w15 = np.array(sampling.candidates(logits, 1.5, 0, 1.0)[1])
    assert w07[0] / w07.sum() > 0.45 > w15[0] / w15.sum()


def check_top_p_keeps_the_shortest_prefix_that_reaches_p(sampling):
    _, p, _ = _example()
    logits = np.log(p).astype(np.float32)
    for top_p, keep in ((0.3, 1), (0.45, 1), (0.5, 2), (0.75, 2), (0.8, 3), (0.95, 4), (1.0, 4)):
        order, w = sampling.candidates(logits, 1.0, 4, top_p)
        assert len(order) == keep, (top_p, order)
        assert np.allclose(np.array(w) / sum(w), p[:keep] / p[:keep].sum(), atol=1e-6)
    with pytest.raises(ValueError):
        sampling.candidates(logits, 1.0, 0, 0.9)


def check_inverse_cdf_frequencies_are_exact_on_a_grid(sampling):
    # n equally spaced u's: candidate i is drawn for the u's inside its CDF interval, so
    # its count is within one of n * p_i
    rng = np.random.default_rng(5)
    x = rng.normal(0, 2, 37).astype(np.float32)
    n = 4000
    for (T, k, tp) in ((1.0, 0, 1.0), (0.8, 10, 1.0), (1.3, 20, 0.9)):
        order, w = sampling.candidates(x, T, k, tp)
        probs = np.array(w) / sum(w)
        counts = {}
        for j in range(n):
            i = sampling.sample(x, T, k, tp, (j + 0.5) / n)
            counts[i] = counts.get(i, 0) + 1
        assert set(counts) <= set(order)
        for i, pi in zip(order, probs):
            assert abs(counts.get(i, 0) - n * pi) <= 1.0 + 1e-9, (i, counts.get(i, 0), n * pi)


def test_top2_example_of_the_page():
    check_top2_example_of_the_page(_sampling)


def test_greedy_is_the_first_largest():
    check_greedy_is_the_first_largest(_sampling)


def test_top_k_order_breaks_ties_by_lower_index():
    check_top_k_order_breaks_ties_by_lower_index(_sampling)


def test_temperature_is_a_power_of_the_distribution():
    check_temperature_is_a_power_of_the_distribution(_sampling)


def test_top_p_keeps_the_shortest_prefix_that_reaches_p():
    check_top_p_keeps_the_shortest_prefix_that_reaches_p(_sampling)


def test_inverse_cdf_frequencies_are_exact_on_a_grid():
    check_inverse_cdf_frequencies_are_exact_on_a_grid(_sampling)
