"""Oracle for the steps on either side of the accept step: the softmax that
turns a pass's logits into probabilities, and the draw of a draft token from
the draft distribution q (float64 and exact integers, numpy).

Test infrastructure only (see the package docstring).

The InvisibleLoRA abstract has a LoRA-off pass propose the next token for
every request and one LoRA-on pass verify the proposals; both passes end in
a distribution over the vocabulary.  The pages give no formula for it; the
reading taken is the usual one for a language model's output layer:

    p(v) = exp(z(v) - max_w z(w)) / sum_u exp(z(u) - max_w z(w))

for a row of logits z (temperature 1; subtracting the maximum changes nothing
mathematically and keeps every exponent at or below 0).  The draft token is
drawn from q with the same exact integer inverse CDF as the accept step's
residual draw (``oracle.accept``): weights Q(q(v)) = floor(q(v) * 2^40),
S = sum of the weights, U = floor(u * 2^32), T = floor(U * S / 2^32), and the
token is the smallest v whose running sum of weights exceeds T.

Readings where the pages are silent:
  * temperature 1, no top-k / top-p truncation;
  * the draw takes the fp32 probabilities the kernel hands to the accept
    step, so that the drawn token and the q the accept step tests it with are
    the same distribution;
  * a uniform >= 1 counts as the largest fp32 below 1, a NaN or negative one
    as 0 (as in the accept step); a row whose weights are all 0 draws token 0.
"""
from __future__ import annotations

import numpy as np

from oracle import accept as OA


def softmax(z):
    """Float64 softmax over the last axis of logits z (any shape [..., V])."""
    z = np.asarray(z, dtype=np.float64)
    m = np.max(z, axis=-1, keepdims=True)
    e = np.exp(z - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def draft_sample(q, u):
    """Draft tokens x[b] ~ q[b] for fp32 probabilities q [B, V] and uniforms
    u [B]: the exact integer inverse CDF of Q(q).  Returns int32 [B]."""
    q = np.asarray(q, dtype=np.float32)
    u, _ = OA._sanitize_uniform(np.asarray(u, dtype=np.float32))
    B = q.shape[0]
    out = np.zeros(B, dtype=np.int32)
    for b in range(B):
        w = OA.quantize(np.clip(np.nan_to_num(q[b], nan=0.0), 0.0, 1.0))
        if int(w.sum(dtype=np.uint64)) == 0:
            out[b] = 0
            continue
        U = int(np.floor(np.float64(u[b]) * 2.0 ** OA.U_BITS))
        out[b] = OA.inverse_cdf_index(w, U)
    return out
