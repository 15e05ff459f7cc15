"""Pins for the FP8 draft-weight oracle (oracle.fp8).

E4M3 is fixed by its definition (sign, 4 exponent bits with bias 7, 3
mantissa bits, saturation at 448 for the conversion used here): the decoded
values of chosen codes worked by hand, every finite code surviving a round
trip, a brute-force nearest-value search with ties to the even mantissa, and
PyTorch's own float8_e4m3fn conversion (a library routine) inside the finite
range.  The per-row quantization is pinned by its largest element landing on
+-448, and the FP8 layer by two facts the mathematics fixes: inputs already on
the E4M3 grid (row maxima 448 times a power of two) give exactly W x, and for
any input the error stays within the format's rounding bound.
"""
import numpy as np
import pytest
import torch

from oracle import fp8 as F


def test_decoded_values_worked_by_hand():
    cases = {
        0x00: 0.0,
        0x01: 2.0 ** -9,            # smallest subnormal: 1/8 * 2^-6
        0x07: 7 * 2.0 ** -9,        # largest subnormal
        0x08: 2.0 ** -6,            # smallest normal: exponent field 1 -> 2^(1-7)
        0x38: 1.0,                  # exponent field 7, mantissa 0
        0x3C: 1.5,                  # mantissa 100 -> 1 + 4/8
        0x40: 2.0,
        0x7E: 448.0,                # exponent field 15, mantissa 110: 1.75 * 2^8
        0x80: -0.0,
        0xB8: -1.0,
        0xFE: -448.0,
    }
    for c, v in cases.items():
        d = F.e4m3_decode(np.array([c], np.uint8))[0]
        assert d == v and np.signbit(d) == np.signbit(v), hex(c)
    assert np.isnan(F.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()


def test_every_finite_code_round_trips():
    c = np.arange(256, dtype=np.uint8)
    v = F.e4m3_decode(c)
    fin = ~np.isnan(v)
    assert fin.sum() == 254
    assert np.array_equal(F.e4m3_round(v[fin].astype(np.float32)), c[fin])


def test_hand_worked_roundings():
    v = np.array([1.0625, 1.1875, 1.0624, 500.0, 1e30, -1e30, 460.0, 2.0 ** -10, 1.5 * 2.0 ** -10, 3 * 2.0 ** -10,
                  np.nan], np.float32)
    expect = [0x38,  # midpoint of 1 and 1.125: ties to the even mantissa 000
              0x3A,  # midpoint of 1.125 (001) and 1.25 (010): to 010
              0x38,  # below the midpoint
              0x7E, 0x7E, 0xFE, 0x7E,  # saturation at 448
              0x00,  # half the smallest subnormal: tie to 0
              0x01,  # 1.5 * 2^-10 rounds up to 2^-9
              0x02,  # 3 * 2^-10 = 1.5 * 2^-9: tie between 1 and 2 (x 2^-9), to the even 2
              0x7F]
    assert F.e4m3_round(v).tolist() == expect


def test_brute_force_nearest_ties_to_even():
    g = np.random.default_rng(0)
    mag = np.exp2(g.uniform(-12, 9.5, 20000)).astype(np.float32)
    sgn = np.where(g.random(20000) < 0.5, -1, 1).astype(np.float32)
    v = (mag * sgn).astype(np.float32)
    pos = np.arange(0x7F, dtype=np.uint8)  # 0x00 .. 0x7E
    vals = F.e4m3_decode(pos)
    got = F.e4m3_round(v)
    for x, c in zip(v.astype(np.float64), got):
        a = min(abs(x), 448.0)
        d = np.abs(vals - a)
        best = np.flatnonzero(d == d.min())
        if len(best) > 1:  # a tie: the code with the even mantissa
            best = [b for b in best if b % 2 == 0]
        want = int(best[0]) | (0x80 if x < 0 else 0)
        assert int(c) == want, (x, hex(int(c)), hex(want))


def test_library_conversion_inside_the_finite_range():
    g = np.random.default_rng(1)
    v = (np.exp2(g.uniform(-12, 8.7, 50000)) * np.where(g.random(50000) < 0.5, -1, 1)).astype(np.float32)
    v = v[np.abs(v) < 448]
    lib = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(F.e4m3_round(v), lib)


def test_row_quantization():
    g = np.random.default_rng(2)
    a = g.standard_normal((6, 300)).astype(np.float32)
    a[3] = 0.0
    codes, s = F.quantize_rows(a)
    assert s[3] == 1.0 and not codes[3].any()
    for r in (0, 1, 2, 4, 5):
        assert s[r] == np.float32(np.max(np.abs(a[r])) / np.float32(448.0))
        i = int(np.argmax(np.abs(a[r])))
        assert codes[r, i] in (0x7E, 0xFE)  # the row's largest magnitude maps to +-448
        assert np.all(np.abs(F.e4m3_decode(codes[r])) <= 448)
    # dequantized values stay within half an E4M3 step of the inputs
    d = F.dequantize_rows(codes, s)
    step = np.maximum(np.abs(a) * 2.0 ** -4, 2.0 ** -10 * s[:, None].astype(np.float64))
    assert np.all(np.abs(d - a) <= step * (1 + 1e-6))


def test_layer_on_grid_inputs_is_exact():
    """W and x whose entries are E4M3 values with each row's maximum exactly
    448 * 2^e: the scales are powers of two, the codes exact, and the FP8
    layer equals W x (plain float64 matmul) exactly."""
    g = np.random.default_rng(3)
    grid = F.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    M, N, K = 5, 7, 64

    def on_grid(R, e):
        c = g.choice(grid, (R, K)) * np.where(g.random((R, K)) < 0.5, -1, 1)
        c[:, 0] = 448.0
        return (c * np.exp2(e)[:, None]).astype(np.float32)

    W = on_grid(N, g.integers(-8, 3, N).astype(np.float64))
    x = on_grid(M, g.integers(-8, 3, M).astype(np.float64))
    Wq, sw = F.quantize_rows(W)
    y = F.draft_layer_fp8(x, Wq, sw)
    assert np.array_equal(y, x.astype(np.float64) @ W.astype(np.float64).T)


def test_layer_error_within_the_format_bound():
    g = np.random.default_rng(4)
    M, N, K = 6, 9, 256
    W = (g.standard_normal((N, K)) / 16).astype(np.float32)
    x = g.standard_normal((M, K)).astype(np.float32)
    W[2, :5] = 0.0
    Wq, sw = F.quantize_rows(W)
    _, sx = F.quantize_rows(x)
    y = F.draft_layer_fp8(x, Wq, sw)
    exact = x.astype(np.float64) @ W.astype(np.float64).T
    dW = np.maximum(np.abs(W) * 2.0 ** -4, 2.0 ** -10 * sw[:, None]) * (1 + 1e-6)
    dx = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * sx[:, None]) * (1 + 1e-6)
    bound = (np.abs(x) + dx) @ dW.T + dx @ np.abs(W).T
    assert np.all(np.abs(y - exact) <= bound + 1e-12)
    # and it is a real approximation, not a bound met trivially
    assert np.max(np.abs(y - exact)) > 0 and np.max(np.abs(y - exact) / bound) > 0.01
