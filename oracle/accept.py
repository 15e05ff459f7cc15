"""Oracle for the per-request accept / resample step (float64 and exact integers).

Test infrastructure only (see the package docstring).

The InvisibleLoRA abstract says one LoRA-on pass verifies every draft token
and that verification keeps the output distribution of plain multi-LoRA
decoding; it gives no rule.  The reading taken here is standard speculative
sampling (Leviathan, Kalman & Matias 2023, "Fast Inference from Transformers
via Speculative Decoding"; Chen et al. 2023, "Accelerating Large Language Model
Decoding with Speculative Sampling"), with every random choice made exact so
that a GPU can reproduce each decision bit for bit:

  inputs per request: target probabilities p_0..p_k (the LoRA-on pass, one per
  verified row), draft probabilities q_0..q_{k-1} (the LoRA-off pass), draft
  tokens x_0..x_{k-1} and uniforms u_0..u_k, all fp32.

  1. For i = 0, 1, ...: keep x_i if u_i * q_i(x_i) < p_i(x_i), the product and
     the comparison taken in float64 (exact: 24 + 24 significant bits).  The
     first failing position is n; if none fails, n = k.
  2. Weights over the vocabulary, in fixed point Q(f) = floor(f * 2^40):
       n < k:  w(v) = max(0, Q(p_n(v)) - Q(q_n(v)))      (residual distribution)
       n = k:  w(v) = Q(p_k(v))                          (bonus token)
  3. S = sum_v w(v) (exact in uint64), U = floor(u_k * 2^32),
     T = floor(U * S / 2^32); emit the smallest v whose running sum of w
     exceeds T.  This is an inverse-CDF draw of w / S.
  4. Output tokens x_0..x_{n-1}, then the drawn token, then -1 padding;
     accepted = n.

Readings where the pages are silent:
  * accept test "u*q < p" (strict); u in [0, 1).
  * the residual in 2^-40 fixed point: its total-variation bias against the
    real-valued residual is below V * 2^-40.
  * if the residual mass S is 0 (reachable only through rounding), draw from
    Q(p_n) instead; if that is 0 too, emit token 0.  Both raise
    STATUS_ZERO_MASS.
  * values read that are NaN or negative count as 0, above 1 as 1; a uniform
    that is NaN or negative counts as 0 and one >= 1 as the largest fp32 below
    1.  Each raises STATUS_BAD_PROB.  A draft token outside [0, V) is rejected
    at its position and raises STATUS_BAD_TOKEN.
"""
from __future__ import annotations

import numpy as np

STATUS_BAD_PROB = 1 << 2
STATUS_BAD_TOKEN = 1 << 3
STATUS_ZERO_MASS = 1 << 4

FIX_BITS = 40
U_BITS = 32
_ONE_MINUS = np.float32(np.nextafter(np.float32(1.0), np.float32(0.0)))


def _sanitize_prob(f):
    f = np.asarray(f, dtype=np.float32)
    bad = np.isnan(f) | (f < 0) | (f > 1)
    g = np.where(np.isnan(f) | (f < 0), np.float32(0), np.where(f > 1, np.float32(1), f))
    return g.astype(np.float32), bad


def _sanitize_uniform(u):
    u = np.asarray(u, dtype=np.float32)
    bad = np.isnan(u) | (u < 0) | (u >= 1)
    g = np.where(np.isnan(u) | (u < 0), np.float32(0), np.where(u >= 1, _ONE_MINUS, u))
    return g.astype(np.float32), bad


def quantize(f) -> np.ndarray:
    """Q(f) = floor(f * 2^40) for fp32 f in [0, 1]; exact (uint64)."""
    return np.floor(np.asarray(f, dtype=np.float32).astype(np.float64) * 2.0 ** FIX_BITS).astype(np.uint64)


def inverse_cdf_index(w_row, U: int) -> int:
    """Smallest v with sum_{v' <= v} w(v') > floor(U * S / 2^32), S = sum w.

    w_row: uint64 weights with S > 0; U in [0, 2^32).
    """
    S = int(np.sum(w_row, dtype=np.uint64))
    T = (int(U) * S) >> U_BITS
    c = np.cumsum(w_row, dtype=np.uint64)
    return int(np.searchsorted(c, np.uint64(T), side="right"))


def acceptance_rate(p_row, q_row) -> float:
    """Closed-form probability that a draft drawn from q is kept: sum_v min(p, q)."""
    return float(np.minimum(np.asarray(p_row, np.float64), np.asarray(q_row, np.float64)).sum())


def accept_decisions(p, q, draft_tok, u):
    """Step 1 for a batch.  Returns (n int64 [B], status)."""
    B, k1, V = p.shape
    k = k1 - 1
    status = 0
    n = np.full(B, k, dtype=np.int64)
    live = np.ones(B, dtype=bool)
    rows = np.arange(B)
    for i in range(k):
        x = np.asarray(draft_tok[:, i], dtype=np.int64)
        bad_tok = live & ((x < 0) | (x >= V))
        if bad_tok.any():
            status |= STATUS_BAD_TOKEN
        xc = np.clip(x, 0, V - 1)
        pi, bp = _sanitize_prob(p[rows, i, xc])
        qi, bq = _sanitize_prob(q[rows, i, xc])
        ui, bu = _sanitize_uniform(u[:, i])
        read = live & ~bad_tok
        if (read & (bp | bq | bu)).any():
            status |= STATUS_BAD_PROB
        keep = ui.astype(np.float64) * qi.astype(np.float64) < pi.astype(np.float64)
        reject = live & (bad_tok | ~keep)
        n[reject] = i
        live &= ~reject
    return n, status


def verify_accept(p, q, draft_tok, u):
    """Whole step.  p fp32 [B, k+1, V], q fp32 [B, k, V], draft_tok int32 [B, k],
    u fp32 [B, k+1].  Returns (out_tok int32 [B, k+1], accepted int32 [B], status)."""
    p = np.asarray(p, dtype=np.float32)
    q = np.asarray(q, dtype=np.float32)
    u = np.asarray(u, dtype=np.float32)
    B, k1, V = p.shape
    k = k1 - 1
    n, status = accept_decisions(p, q, draft_tok, u)
    out = np.full((B, k1), -1, dtype=np.int32)
    uk, bu = _sanitize_uniform(u[:, k])
    if bu.any():
        status |= STATUS_BAD_PROB
    for b in range(B):
        nb = int(n[b])
        out[b, :nb] = draft_tok[b, :nb]
        pn, bp = _sanitize_prob(p[b, nb])
        if bp.any():
            status |= STATUS_BAD_PROB
        if nb < k:
            qn, bq = _sanitize_prob(q[b, nb])
            if bq.any():
                status |= STATUS_BAD_PROB
            w = np.maximum(quantize(pn).astype(np.int64) - quantize(qn).astype(np.int64), 0).astype(np.uint64)
            if int(w.sum(dtype=np.uint64)) == 0:
                status |= STATUS_ZERO_MASS
                w = quantize(pn)
        else:
            w = quantize(pn)
        if int(w.sum(dtype=np.uint64)) == 0:
            status |= STATUS_ZERO_MASS
            tok = 0
        else:
            U = int(np.floor(np.float64(uk[b]) * 2.0 ** U_BITS))
            tok = inverse_cdf_index(w, U)
        out[b, nb] = tok
    return out, n.astype(np.int32), status
