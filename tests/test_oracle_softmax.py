"""Pins for the softmax and draft-draw oracle (oracle.softmax).

Each test checks the oracle against a fact the mathematics fixes, not
against a retyped formula: constant logits give 1/V, two tokens give the
logistic function, adding a constant to every logit changes nothing, the
ratio of two probabilities is exp of the logit difference, a dominant logit
gives (nearly) all the mass, and the draw's frequencies over every value of
U are the weights' exact shares.
"""
import math

import numpy as np
import pytest

from oracle import accept as OA
from oracle import softmax as OS


def test_constant_logits_are_uniform():
    for V in (1, 2, 7, 1000):
        p = OS.softmax(np.full((3, V), 2.5))
        assert np.allclose(p, 1.0 / V, rtol=0, atol=1e-15)


def test_two_tokens_follow_the_logistic_function():
    for a, b in [(0.0, 0.0), (1.0, -2.0), (30.0, 29.5), (-7.25, 3.0)]:
        p = OS.softmax(np.array([a, b]))
        assert p[0] == pytest.approx(1.0 / (1.0 + math.exp(b - a)), rel=1e-14)
        assert p[1] == pytest.approx(1.0 / (1.0 + math.exp(a - b)), rel=1e-14)


def test_shift_invariance_and_ratio():
    g = np.random.default_rng(3)
    z = g.standard_normal((5, 64)) * 4
    p = OS.softmax(z)
    assert np.allclose(OS.softmax(z + 123.0), p, rtol=1e-13, atol=0)
    assert np.allclose(p.sum(-1), 1.0, atol=1e-14)
    i, j = 3, 17
    assert np.allclose(p[:, i] / p[:, j], np.exp(z[:, i] - z[:, j]), rtol=1e-12)


def test_dominant_logit_takes_the_mass():
    z = np.zeros((1, 50))
    z[0, 7] = 60.0  # every other entry weighs exp(-60) < 1e-26
    p = OS.softmax(z)
    assert p[0, 7] == pytest.approx(1.0, abs=1e-24) and p[0].argmax() == 7
    assert np.all(p[0, np.arange(50) != 7] == pytest.approx(math.exp(-60.0) / (1 + 49 * math.exp(-60.0)), rel=1e-12))


def test_draft_sample_frequencies_are_exact():
    """Over the 2^24 uniforms u = j / 2^24 (each exact in fp32) the draw is
    monotone in j, and token v takes within one of Q(q(v)) 2^24 / S of them
    (its exact share), none when Q(q(v)) = 0.  Found by bisection on j."""
    q = np.array([[0.5, 0.0, 0.25, 0.1, 0.15]], np.float32)
    w = OA.quantize(q[0])
    S = int(w.sum())

    def draw(j):
        return int(OS.draft_sample(q, np.array([np.float32(j / 2 ** 24)], np.float32))[0])

    starts = []
    for v in range(len(w) + 1):
        lo, hi = 0, 2 ** 24
        while lo < hi:
            mid = (lo + hi) // 2
            if draw(mid) >= v:
                hi = mid
            else:
                lo = mid + 1
        starts.append(lo)
    counts = np.diff(starts)
    for v in range(len(w)):
        assert abs(counts[v] - int(w[v]) * 2 ** 24 / S) <= 1.0, (v, counts[v])
        assert (counts[v] == 0) == (int(w[v]) == 0)


def test_draft_sample_hand_worked():
    # Q(q) = [2^39, 0, 2^38, 2^37, 2^37], S = 2^40; u = 0.5: U = 2^31, T = 2^39,
    # cumsum = [2^39, 2^39, 3 2^38, 7 2^37, 2^40]; the first above T is index 2.
    q = np.array([[0.5, 0.0, 0.25, 0.125, 0.125]], np.float32)
    assert OS.draft_sample(q, np.array([0.5], np.float32)).tolist() == [2]
    # u = 0: T = 0, the first nonzero weight: token 0.  u = 1.5 counts as 1 - 2^-24: the last nonzero weight.
    assert OS.draft_sample(q, np.array([0.0], np.float32)).tolist() == [0]
    assert OS.draft_sample(q, np.array([1.5], np.float32)).tolist() == [4]
    # a zero row draws token 0
    assert OS.draft_sample(np.zeros((1, 4), np.float32), np.array([0.3], np.float32)).tolist() == [0]


def test_draft_sample_follows_q():
    """Chi-square on V = 6: draws from one fp32 q over 60000 uniforms."""
    from scipy import stats
    g = np.random.default_rng(4)
    q = OS.softmax(g.standard_normal(6) * 1.5).astype(np.float32)
    T = 60000
    u = g.random(T, dtype=np.float32)
    x = OS.draft_sample(np.broadcast_to(q, (T, 6)), u)
    counts = np.bincount(x, minlength=6)
    q64 = q.astype(np.float64)
    assert stats.chisquare(counts, q64 / q64.sum() * T).pvalue > 0.01
