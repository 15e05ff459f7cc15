"""Oracle for the run-time draft gate (exact rationals and floats, host only).

Test infrastructure only (see the package docstring).

The InvisibleLoRA abstract has a run-time gate that skips drafting on steps
where the adapter cost cannot repay a draft pass.  The pages give no formula;
the reading taken is the usual cost model of speculative decoding (Leviathan,
Kalman & Matias 2023): with draft length k and each draft kept with
probability alpha independently of the others (until the first rejection),
the number n of kept drafts has

    P(n) = alpha^n (1 - alpha)  for n < k,    P(k) = alpha^k,

and a cycle emits n + 1 tokens (the kept drafts and the drawn token), so the
expected tokens per cycle are E(alpha, k) = sum_n (n + 1) P(n).  A cycle with
k drafts costs t_cycle[k] (k LoRA-off passes, one LoRA-on pass over k + 1
rows per request, the accept step); plain multi-LoRA decoding emits one token
per request per LoRA-on pass of cost t_plain.  The gate drafts with the k
that maximises E(alpha, k) / t_cycle[k] if that rate beats 1 / t_plain, and
skips drafting (k = 0) otherwise.

The acceptance rate is estimated from the accept step's counts: the maximum
of the likelihood prod_b P(n_b) is alpha = sum n_b / (sum n_b + #{b : n_b < k}).
"""
from __future__ import annotations

from fractions import Fraction


def expected_tokens(alpha, k: int):
    """E(alpha, k) = sum over n of (n + 1) P(n), by enumeration of the
    distribution (exact when alpha is a Fraction)."""
    total = 0
    for n in range(k + 1):
        pn = alpha ** n * ((1 - alpha) if n < k else 1)
        total += (n + 1) * pn
    return total


def draft_gate(t_cycle: dict, t_plain: float, alpha: float):
    """(k, gain): the draft length with the best token rate, or 0 when plain
    decoding is faster; gain = best rate * t_plain (tokens per t_plain)."""
    best_k, best_rate = 0, 1.0 / t_plain
    for k in sorted(t_cycle):
        rate = expected_tokens(alpha, k) / t_cycle[k]
        if rate > best_rate:
            best_k, best_rate = k, rate
    return best_k, best_rate * t_plain


def estimate_acceptance(accepted, k: int) -> float:
    """Maximum-likelihood alpha from per-request kept-draft counts n_b in [0, k]."""
    s = sum(int(n) for n in accepted)
    short = sum(1 for n in accepted if int(n) < k)
    if s + short == 0:
        return 0.0
    return float(Fraction(s, s + short))
