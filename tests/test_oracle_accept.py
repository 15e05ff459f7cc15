"""Pins for the accept/resample oracle.

The distribution tests check the property the InvisibleLoRA abstract states
(verification keeps the target distribution) by brute force on a tiny
vocabulary; the closed-form acceptance rate sum_v min(p, q) is the one derived
by Leviathan et al. (2023); the other tests are worked examples, special
cases and exactness properties of the integer draw.
"""
import json
import os

import numpy as np
import pytest
from scipy import stats

from oracle import accept as OA
import workloads as WL

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _arr(x, dt):
    return np.asarray(x, dtype=dt)


def test_hand_worked_examples():
    g = json.load(open(os.path.join(GOLDEN, "accept_hand_example.json")))
    for c in g["cases"]:
        out, acc, st = OA.verify_accept(_arr(c["p"], np.float32), _arr(c["q"], np.float32),
                                        _arr(c["draft_tok"], np.int32), _arr(c["u"], np.float32))
        assert st == c.get("status", 0), c["why"]
        assert out.tolist() == c["out_tok"], c["why"]
        assert acc.tolist() == c["accepted"], c["why"]


def _tiny_dist(g, V, n, alpha=1.5):
    d = g.dirichlet(np.full(V, alpha), size=n).astype(np.float32)
    return d


def _trials(p1, q1, k, T, seed):
    """Broadcast one request's distributions over T trials with fresh randomness."""
    g = np.random.default_rng(seed)
    V = p1.shape[-1]
    p = np.broadcast_to(p1, (T, k + 1, V)).copy()
    q = np.broadcast_to(q1, (T, k, V)).copy()
    tok = np.empty((T, k), np.int32)
    for i in range(k):
        qd = q1[i].astype(np.float64)
        tok[:, i] = g.choice(V, size=T, p=qd / qd.sum())
    u = g.random((T, k + 1), dtype=np.float32)
    return p, q, tok, u


def _chi2_pvalue(samples, probs):
    V = probs.shape[0]
    counts = np.bincount(samples, minlength=V)
    expected = probs / probs.sum() * samples.size
    keep = expected >= 5
    obs = np.append(counts[keep], counts[~keep].sum())
    exp = np.append(expected[keep], expected[~keep].sum())
    if exp[-1] == 0:
        obs, exp = obs[:-1], exp[:-1]
    return stats.chisquare(obs, exp).pvalue


@pytest.mark.parametrize("k", [1, 2])
def test_output_follows_target_distribution(k):
    g = np.random.default_rng(100 + k)
    V, T = 8, 60000
    p1 = _tiny_dist(g, V, k + 1)
    q1 = _tiny_dist(g, V, k)
    p, q, tok, u = _trials(p1, q1, k, T, seed=200 + k)
    out, acc, st = OA.verify_accept(p, q, tok, u)
    assert st == 0
    for i in range(k + 1):
        reached = acc >= i          # position i is emitted iff the first i drafts were kept
        pv = _chi2_pvalue(out[reached, i], p1[i].astype(np.float64))
        assert pv > 0.01, (k, i, pv)
    # acceptance rate at position 0 against the closed form
    alpha = OA.acceptance_rate(p1[0], q1[0])
    rate = np.mean(acc >= 1)
    half = 3.29 * np.sqrt(alpha * (1 - alpha) / T)
    assert abs(rate - alpha) <= half, (rate, alpha)


def test_sampling_from_draft_distribution_would_fail():
    """Guard on the test's power: emitting the draft token always (no
    correction) gives a clearly different distribution at this size."""
    g = np.random.default_rng(7)
    V, T = 8, 60000
    p1 = _tiny_dist(g, V, 2)
    q1 = _tiny_dist(g, V, 1)
    _, _, tok, _ = _trials(p1, q1, 1, T, seed=8)
    assert _chi2_pvalue(tok[:, 0], p1[0].astype(np.float64)) < 1e-6


def test_q_equal_p_accepts_everything():
    p, q, tok, u = WL.accept_inputs(1000, 16, 3, sigma=0.3, seed=3)
    q = p[:, :3].copy()
    g = np.random.default_rng(0)
    for b in range(16):
        for i in range(3):
            c = np.cumsum(q[b, i].astype(np.float64))
            tok[b, i] = min(int(np.searchsorted(c, g.random() * c[-1], side="right")), 999)
    out, acc, st = OA.verify_accept(p, q, tok, u)
    assert st == 0 and (acc == 3).all()
    assert np.array_equal(out[:, :3], tok)


def test_one_hot_target_always_emits_its_token():
    g = np.random.default_rng(5)
    V, B, k = 16, 200, 2
    vstar = 9
    p = np.zeros((B, k + 1, V), np.float32)
    p[:, :, vstar] = 1.0
    q = _tiny_dist(g, V, B * k).reshape(B, k, V)
    tok = g.integers(0, V, (B, k)).astype(np.int32)
    u = g.random((B, k + 1), dtype=np.float32)
    out, acc, st = OA.verify_accept(p, q, tok, u)
    assert st == 0
    for b in range(B):
        assert (out[b, :acc[b] + 1] == vstar).all()
        assert (out[b, acc[b] + 1:] == -1).all()


def test_inverse_cdf_frequencies_are_exact():
    """Over all 2^32 values of U, token v is drawn for either floor or ceil of
    w(v) 2^32 / S of them, and never when w(v) = 0.  The first U drawing each
    token is found by bisection on the (monotone) draw."""
    for w in ([3, 0, 5, 1], [1, 1, 1, 1], [0, 0, 7, 0], [2**40, 2**39, 0, 12345]):
        w = np.asarray(w, np.uint64)
        S = int(w.sum())
        starts = []
        for v in range(len(w) + 1):
            lo, hi = 0, 2**32          # smallest U with draw(U) >= v
            while lo < hi:
                mid = (lo + hi) // 2
                if OA.inverse_cdf_index(w, mid) >= v:
                    hi = mid
                else:
                    lo = mid + 1
            starts.append(lo)
        counts = np.diff(starts)
        for v in range(len(w)):
            exact = int(w[v]) * 2**32 / S
            assert abs(counts[v] - exact) < 1.0, (w, v, counts[v], exact)
            assert (counts[v] == 0) == (int(w[v]) == 0)
        assert OA.inverse_cdf_index(w, 0) == int(np.nonzero(w)[0][0])
        assert OA.inverse_cdf_index(w, 2**32 - 1) == int(np.nonzero(w)[0][-1])


def test_fixed_point_residual_is_close_to_the_real_residual():
    g = np.random.default_rng(9)
    V = 64
    for _ in range(20):
        p = g.dirichlet(np.ones(V)).astype(np.float32)
        q = g.dirichlet(np.ones(V)).astype(np.float32)
        w = np.maximum(OA.quantize(p).astype(np.int64) - OA.quantize(q).astype(np.int64), 0).astype(np.float64)
        real = np.maximum(p.astype(np.float64) - q.astype(np.float64), 0)
        tv = 0.5 * np.abs(w / w.sum() - real / real.sum()).sum()
        assert tv <= V * 2.0**-40 / real.sum()


def test_quantize_is_exact():
    f = np.array([0.0, 1.0, 0.5, 2.0**-40, 2.0**-41, 0.1, np.float32(1) - np.float32(2**-24)], np.float32)
    qv = OA.quantize(f)
    for fi, qi in zip(f, qv):
        from fractions import Fraction
        assert int(qi) == int(Fraction(float(fi)) * 2**40 // 1)


def test_invalid_inputs_raise_status_and_stay_defined():
    p = np.array([[[0.5, 0.5, 0.0, 0.0], [0.25, 0.25, 0.25, 0.25]]], np.float32)
    q = np.array([[[0.25, 0.25, 0.25, 0.25]]], np.float32)
    # draft token out of range: rejected at 0
    out, acc, st = OA.verify_accept(p, q, np.array([[7]], np.int32), np.array([[0.1, 0.5]], np.float32))
    assert st & OA.STATUS_BAD_TOKEN and acc[0] == 0 and out[0, 0] in (0, 1)
    # NaN probability in a row that is read
    p2 = p.copy()
    p2[0, 0, 3] = np.nan
    _, _, st = OA.verify_accept(p2, q, np.array([[3]], np.int32), np.array([[0.1, 0.5]], np.float32))
    assert st & OA.STATUS_BAD_PROB
    # p = q exactly on the rejected row is impossible to reject; force zero mass with p = 0 row
    pz = np.zeros((1, 2, 4), np.float32)
    qz = np.zeros((1, 1, 4), np.float32)
    out, acc, st = OA.verify_accept(pz, qz, np.array([[1]], np.int32), np.array([[0.1, 0.5]], np.float32))
    assert st & OA.STATUS_ZERO_MASS and out[0, 0] == 0 and acc[0] == 0


def test_accept_inputs_hit_the_acceptance_band():
    p, q, tok, u = WL.accept_inputs(WL.LLAMA3_VOCAB, 8, 1, seed=0)
    rates = [OA.acceptance_rate(p[b, 0], q[b, 0]) for b in range(8)]
    assert 0.92 <= float(np.mean(rates)) <= 0.97
    assert np.allclose(p.sum(-1), 1.0, atol=1e-4) and np.allclose(q.sum(-1), 1.0, atol=1e-4)
