"""The fixed-point quantisation Q(f) = floor(f * 2^40) as the streaming accept
kernel computes it, with FP32 fused multiply-adds rounding toward minus
infinity instead of a float-to-integer conversion:

    y = RD(f * 2^17 + 2^23)               -> 2^23 + hi,  hi = floor(f * 2^17)
    c = RN(-(y - 2^23) * 2^23 + 2^23)      exact: (1 - hi) * 2^23
    z = RD(f * 2^40 + c)                  -> 2^23 + lo,  lo = floor(f * 2^40 - hi * 2^23)
    Q = hi * 2^23 + lo

Each rounding is emulated exactly with rationals (round to the float32 grid),
so this checks the identity itself, for every f in [0, 1] sampled here and
the edge cases, together with the two facts the residual sums use: Q is
monotone, so sum max(Q(p) - Q(q), 0) = sum Q(p) - sum Q(min(p, q))."""
import math
from fractions import Fraction as Fr

import numpy as np


def _ulp(x):
    e = math.floor(math.log2(x))
    while Fr(2) ** e > x:
        e -= 1
    while Fr(2) ** (e + 1) <= x:
        e += 1
    return Fr(2) ** (e - 23)


def _round_down_f32(x):
    """Largest float32 <= x (x > 0, normal range)."""
    u = _ulp(x)
    return (x // u) * u


def _exact_f32(x):
    assert Fr(float(np.float32(float(x)))) == x, "not representable"
    return x


def q_fma(f):
    f = Fr(float(np.float32(f)))
    y = _round_down_f32(f * 2 ** 17 + 2 ** 23)
    c = _exact_f32(-(y - 2 ** 23) * 2 ** 23 + 2 ** 23)
    z = _round_down_f32(f * 2 ** 40 + c)
    hi, lo = y - 2 ** 23, z - 2 ** 23
    assert hi.denominator == 1 and lo.denominator == 1 and 0 <= lo < 2 ** 23
    return int(hi) * 2 ** 23 + int(lo)


def q_def(f):
    return math.floor(Fr(float(np.float32(f))) * 2 ** 40)


def _samples():
    g = np.random.default_rng(7)
    edge = [0.0, 1.0, 2.0 ** -17, 2.0 ** -40, 2.0 ** -41, 1e-45, 2.0 ** -126,
            float(np.nextafter(np.float32(1), np.float32(0))),
            float(np.nextafter(np.float32(2 ** -17), np.float32(0))),
            float(np.nextafter(np.float32(2 ** -17), np.float32(1))),
            float(np.nextafter(np.float32(2 ** -40), np.float32(1)))]
    uni = g.random(3000).astype(np.float32)
    small = np.exp(-g.random(3000) * 60).astype(np.float32)  # softmax-like tails down to e^-60
    return [np.float32(v) for v in edge] + list(uni) + list(small)


def test_fma_construction_equals_floor():
    for f in _samples():
        assert q_fma(f) == q_def(f), float(f)


def test_residual_sum_identity():
    g = np.random.default_rng(8)
    p = np.exp(-g.random(500) * 30).astype(np.float32)
    q = np.exp(-g.random(500) * 30).astype(np.float32)
    lhs = sum(max(q_def(a) - q_def(b), 0) for a, b in zip(p, q))
    rhs = sum(q_def(a) for a in p) - sum(q_def(min(a, b)) for a, b in zip(p, q))
    assert lhs == rhs
    for a, b in zip(p[:100], q[:100]):  # monotone: the order of floats carries over to Q
        assert (q_def(a) <= q_def(b)) == (a <= b) or q_def(a) == q_def(b)
