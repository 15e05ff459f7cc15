"""Pins for the draft-gate oracle (oracle.gate) and its C implementation.

The oracle enumerates the acceptance distribution; the pins are facts the
mathematics fixes without that enumeration: the geometric-series closed form
(1 - alpha^(k+1)) / (1 - alpha), the limits alpha = 0 (one token) and
alpha = 1 (k + 1 tokens), a Monte Carlo run of the accept rule itself, and the
likelihood's maximum found by a grid search.  The library's host functions
(no GPU needed) are then checked against the oracle.
"""
import ctypes
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import gate as OG


def test_closed_form_of_the_geometric_series():
    for a in (Fraction(0), Fraction(1, 3), Fraction(9, 10), Fraction(97, 100)):
        for k in range(0, 9):
            closed = (1 - a ** (k + 1)) / (1 - a)
            assert OG.expected_tokens(a, k) == closed


def test_limits():
    for k in range(0, 9):
        assert OG.expected_tokens(Fraction(0), k) == 1
        assert OG.expected_tokens(Fraction(1), k) == k + 1
    assert OG.expected_tokens(Fraction(1, 2), 1) == Fraction(3, 2)  # 1 + alpha


def test_monte_carlo_of_the_accept_rule():
    """Simulate: keep drafts while a uniform is below alpha, emit kept + 1."""
    g = np.random.default_rng(0)
    alpha, k, T = 0.8, 4, 200000
    u = g.random((T, k))
    kept = np.argmin(np.concatenate([u < alpha, np.zeros((T, 1), bool)], axis=1), axis=1)
    tokens = kept + 1
    e = OG.expected_tokens(alpha, k)
    assert abs(tokens.mean() - e) < 4 * tokens.std() / np.sqrt(T)


def test_gate_decisions():
    # drafting k = 2 costs 1.5 plain steps and yields 1 + a + a^2 tokens
    assert OG.draft_gate({2: 1.5}, 1.0, 0.9)[0] == 2            # 2.71 tokens for 1.5 > 1 token for 1
    assert OG.draft_gate({2: 3.0}, 1.0, 0.5)[0] == 0            # 1.75 tokens for 3 < 1 token for 1
    k, gain = OG.draft_gate({1: 1.2, 2: 1.4, 4: 1.9}, 1.0, 0.95)
    rates = {1: 1.95 / 1.2, 2: (1 + 0.95 + 0.95 ** 2) / 1.4, 4: (1 - 0.95 ** 5) / 0.05 / 1.9}
    assert k == max(rates, key=rates.get) and gain == pytest.approx(max(rates.values()))


def test_acceptance_estimate_maximises_the_likelihood():
    counts = [4, 4, 2, 4, 0, 3, 4, 4, 1, 4]
    k = 4
    a_hat = OG.estimate_acceptance(counts, k)

    def loglik(a):
        return sum(n * np.log(a) + (np.log(1 - a) if n < k else 0.0) for n in counts)

    grid = np.linspace(0.01, 0.99, 9801)
    assert abs(grid[np.argmax([loglik(a) for a in grid])] - a_hat) < 1e-4
    assert OG.estimate_acceptance([k] * 5, k) == 1.0 and OG.estimate_acceptance([0] * 5, k) == 0.0


# ---- the library's host implementation (loads without a GPU) ----

@pytest.fixture(scope="module")
def lib():
    import speculative_lora_decoding_gb300 as ml
    if not os.path.exists(ml.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return ml.library()


def test_library_gate_matches_oracle(lib):
    g = np.random.default_rng(3)
    for _ in range(200):
        alpha = float(g.random())
        kmax = int(g.integers(1, 9))
        t_plain = float(g.random() + 0.1)
        t = (ctypes.c_double * (kmax + 1))(*([0.0] + [float(t_plain * (0.8 + 0.4 * j * g.random())) for j in range(1, kmax + 1)]))
        gain = ctypes.c_double(0.0)
        k = lib.mlora_draft_gate(t, kmax, t_plain, alpha, ctypes.byref(gain))
        k_ref, gain_ref = OG.draft_gate({j: t[j] for j in range(1, kmax + 1)}, t_plain, alpha)
        assert k == k_ref and gain.value == pytest.approx(gain_ref, rel=1e-12)
        for j in range(0, kmax + 1):
            assert lib.mlora_expected_tokens(alpha, j) == pytest.approx(float(OG.expected_tokens(alpha, j)), rel=1e-12)
    counts = (ctypes.c_int32 * 6)(4, 4, 2, 0, 4, 3)
    assert lib.mlora_estimate_acceptance(counts, 6, 4) == pytest.approx(OG.estimate_acceptance(list(counts), 4))
    assert lib.mlora_draft_gate(None, 4, 1.0, 0.5, None) == -1  # invalid arguments
