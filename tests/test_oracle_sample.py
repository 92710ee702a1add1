"""Pins for the oracle's sampling step after the output head (top-k, temperature,
top-p, draw): argmax and plain-softmax special cases, closed forms, ties.  CPU only."""
import math

import numpy as np
import pytest
from scipy.special import softmax


def test_top_k_one_is_the_argmax(orc):
    rng = np.random.default_rng(0)
    for V in (1, 7, 1000):
        lg = rng.standard_normal(V).astype(np.float32) * 3
        for u in (0.0, 0.5, 0.999):
            idx, m = orc.sample(lg, 1.0, 1, 0.95, u)
            assert idx == int(np.argmax(lg)) and m == 1


def test_no_truncation_follows_the_softmax_cdf(orc):
    # top_k = V and top_p = 1: the draw inverts the softmax CDF over the sorted logits
    rng = np.random.default_rng(1)
    V = 6
    for T in (1.0, 0.5, 2.0):
        lg = rng.standard_normal(V).astype(np.float32)
        order = np.argsort(-lg, kind="stable")
        cdf = np.cumsum(softmax(lg[order].astype(np.float64) / T))
        for u in np.linspace(0.0, 0.999, 97):
            if np.min(np.abs(cdf - u)) < 1e-9:
                continue
            want = order[int(np.searchsorted(cdf, u, side="right"))]
            idx, m = orc.sample(lg, T, V, 1.0, u)
            assert idx == want and m == V


def test_closed_form(orc):
    # p = 0.4, 0.3, 0.2, 0.1 (sorted).  top_p 0.65: the prefix {0.4, 0.3} reaches it,
    # q = 4/7, 3/7.  Temperature 2 takes square roots before normalising.
    lg = np.log(np.array([0.1, 0.2, 0.3, 0.4])).astype(np.float32)
    assert orc.sample(lg, 1.0, 4, 0.65, 0.5) == (3, 2)
    assert orc.sample(lg, 1.0, 4, 0.65, 4 / 7 + 1e-6) == (2, 2)
    assert orc.sample(lg, 1.0, 4, 0.65, 0.999) == (2, 2)
    assert orc.sample(lg, 1.0, 4, 0.7 + 1e-6, 0.9) == (1, 3)       # 0.4 + 0.3 falls short
    assert orc.sample(lg, 1.0, 4, 1.0, 0.95) == (0, 4)
    assert orc.sample(lg, 1.0, 2, 0.95, 0.6) == (2, 2)              # top-2, both kept
    s = np.sqrt([0.4, 0.3, 0.2, 0.1]); s /= s.sum()                 # temperature 2
    m = int(np.searchsorted(np.cumsum(s), 0.6) + 1)
    q = np.cumsum(s[:m]) / s[:m].sum()
    u = (q[0] + q[1]) / 2
    assert orc.sample(lg, 2.0, 4, 0.6, u) == (2, m)


def test_ties_and_minus_infinity(orc):
    # equal logits: the lowest indices are the candidates, with equal probabilities
    lg = np.full(10, 1.5, np.float32)
    assert orc.sample(lg, 1.0, 3, 0.5, 0.4) == (0, 2)
    assert orc.sample(lg, 1.0, 3, 0.5, 0.6) == (1, 2)
    assert orc.sample(lg, 1.0, 3, 1.0, 0.9) == (2, 3)
    # NaN reads as -inf; all -inf draws the first candidate
    lg = np.array([np.nan, -np.inf, 0.0, np.nan], np.float32)
    assert orc.sample(lg, 1.0, 2, 0.95, 0.99)[0] == 2
    assert orc.sample(np.full(4, -np.inf, np.float32), 1.0, 3, 0.95, 0.7) == (0, 1)


@pytest.mark.parametrize("seed", range(4))
def test_kept_prefix_is_the_shortest(orc, seed):
    rng = np.random.default_rng(10 + seed)
    lg = (rng.standard_normal(500) * 2).astype(np.float32)
    for k, p in [(20, 0.95), (50, 0.5), (5, 0.99)]:
        order = np.argsort(-lg, kind="stable")[:k]
        pr = softmax(lg[order].astype(np.float64))
        cum = np.cumsum(pr)
        if np.min(np.abs(cum - p)) < 1e-9:
            continue
        want_m = min(k, int(np.searchsorted(cum, p) + 1))
        idx, m = orc.sample(lg, 1.0, k, p, 0.0)
        assert m == want_m and idx == order[0]


def test_plus_infinity_takes_all_the_mass(orc):
    # softmax's limit: a +inf logit has probability 1; with several, the lowest index
    # (rank 0 in the top-k's tie order) is drawn, whatever the uniform
    lg = np.array([0.5, np.inf, 3.0, np.inf, -1.0], np.float32)
    for u in (0.0, 0.5, 0.999):
        assert orc.sample(lg, 1.0, 4, 0.95, u) == (1, 1)
    lg = np.array([2.0, np.nan, np.inf], np.float32)
    assert orc.sample(lg, 0.7, 3, 0.5, 0.9) == (2, 1)
