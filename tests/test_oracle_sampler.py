"""Pins of the sampler oracle against closed forms and a library softmax."""

import math

import numpy as np
import pytest
from scipy.special import softmax

from oracle import sampler as S


def _token_fractions(vals, temperature, top_p, n=200_001):
    """Fraction of a fine grid of u in [0, 1) that draws each candidate (inverse CDF)."""
    idx = np.arange(len(vals))
    us = (np.arange(n) + 0.5) / n
    hits = np.zeros(len(vals))
    for u in us:
        hits[S.sample_topk(vals, idx, temperature, top_p, u)] += 1
    return hits / n


def test_inverse_cdf_matches_library_softmax():
    rng = np.random.default_rng(5)
    vals = np.sort(rng.normal(0, 1.5, 6))[::-1].astype(np.float32)
    for t in (0.6, 1.0, 2.5):
        p = softmax(vals.astype(np.float64) / t)
        frac = _token_fractions(vals, t, 1.0, n=50_001)
        assert np.allclose(frac, p, atol=1e-4), (t, frac, p)


def test_nucleus_cut_closed_form():
    # probabilities 0.5, 0.3, 0.15, 0.05 at T = 0.6: top_p 0.9 keeps the first three
    p = np.array([0.5, 0.3, 0.15, 0.05])
    t = 0.6
    vals = (np.log(p) * t).astype(np.float64)
    frac = _token_fractions(vals, t, 0.9, n=40_001)
    want = np.array([0.5, 0.3, 0.15, 0.0]) / 0.95
    assert np.allclose(frac, want, atol=1e-4)
    # top_p 0.8 (0.5 + 0.3 reaches it exactly): the crossing candidate stays, the rest go
    frac = _token_fractions(vals, t, 0.79, n=40_001)
    assert np.allclose(frac, np.array([0.5, 0.3, 0.0, 0.0]) / 0.8, atol=1e-4)


def test_hand_worked_draws():
    # logits 2, 1, 0 at T = 1: e = e^0, e^-1, e^-2 relative to the first; cumulative shares
    # 0.6652, 0.9100, 1.0 of the total 1 + e^-1 + e^-2 = 1.5032
    vals, idx = [2.0, 1.0, 0.0], [70, 71, 72]
    assert S.sample_topk(vals, idx, 1.0, 1.0, 0.50) == 70
    assert S.sample_topk(vals, idx, 1.0, 1.0, 0.70) == 71
    assert S.sample_topk(vals, idx, 1.0, 1.0, 0.95) == 72
    shares = np.cumsum([1.0, math.exp(-1), math.exp(-2)]) / (1 + math.exp(-1) + math.exp(-2))
    assert abs(shares[0] - 0.66524) < 1e-5 and abs(shares[1] - 0.90997) < 1e-5


@pytest.mark.parametrize("u", [0.0, 0.3, 0.999999])
def test_greedy_limits(u):
    vals, idx = [3.0, 2.9, 1.0], [5, 6, 7]
    assert S.sample_topk(vals, idx, 0.0, 0.95, u) == 5          # temperature 0: greedy
    assert S.sample_topk(vals, idx, 0.6, 1e-12, u) == 5         # nucleus of one
    assert S.sample_topk([3.0, 2.0], idx[:2], 1e-3, 1.0, u) == 5  # near-zero temperature


def test_margin_flags_boundaries():
    vals = [1.0, 0.0]
    e = [1.0, math.exp(-1.0)]
    u_edge = e[0] / sum(e)
    assert S.decision_margin(vals, 1.0, 1.0, u_edge) < 1e-12
    assert S.decision_margin(vals, 1.0, 1.0, 0.3) > 1e-3
