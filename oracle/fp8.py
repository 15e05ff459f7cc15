"""Oracle for the draft pass on FP8 base weights (numpy; exact rounding to
E4M3 from its definition, float64 sums).

Test infrastructure only (see the package docstring).

The pages list quantization of the base weights to 8 bits (INT8 or FP8) as a
serving optimisation that goes with LoRA ("LoRA Inference" glossary, the
serving-optimisations list and the quantization paragraph).  InvisibleLoRA's
draft pass runs the base model alone (LoRA off), so its weights can be an FP8
copy of W: half the bytes of the HBM-bound draft.  Drafts only propose
tokens; the LoRA-on verify pass (bf16) and the accept step decide what is
emitted, so FP8 drafts change the acceptance rate, never the output
distribution.  The readings taken where the pages say nothing:

  * Format E4M3 (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
    largest finite 448, smallest normal 2^-6, subnormals down to 2^-9; no
    infinities; code 0x7F / 0xFF is NaN).  Rounding to nearest, ties to an
    even mantissa; magnitudes above 448 saturate to 448.
  * One fp32 scale per row: s = amax / 448 (fp32 division) with amax the
    largest |value| of the row; the codes are e4m3(v / s) of the fp32
    quotient.  A row of zeros gets s = 1 and zero codes.  Inputs are finite
    (bf16 weights and activations).  W is quantized per output row (offline),
    the activations x per token row (every call).
  * The draft layer output is y[m, n] = bf16(s_x[m] s_w[n] sum_k Wq[n, k] xq[m, k])
    with Wq, xq the decoded codes; the oracle gives the float64 value before
    the bf16 rounding.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
NAN_CODE = 0x7F


def e4m3_decode(codes) -> np.ndarray:
    """Float64 value of each E4M3 code (NaN for 0x7F and 0xFF)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = sign * (1.0 + m / 8.0) * np.exp2(e - 7.0)
    sub = sign * (m / 8.0) * 2.0 ** -6
    v = np.where(e == 0, sub, normal)
    return np.where((c & 0x7F) == 0x7F, np.nan, v)


def e4m3_round(v) -> np.ndarray:
    """E4M3 codes of fp32 values: nearest, ties to even, saturating at 448;
    NaN gives the NaN code.  Exact: works on the float64 value of each fp32
    input; the binade's spacing is a power of two, so the quotient by it and
    the tie test are exact."""
    x = np.asarray(v, dtype=np.float32).astype(np.float64)
    sign = np.where(np.signbit(x), 0x80, 0).astype(np.int64)
    a = np.abs(np.nan_to_num(x, nan=0.0))
    # binade exponent e with 2^e <= a < 2^(e+1); the subnormals share 2^-6's spacing
    _, p = np.frexp(a)
    e = np.maximum(p - 1, -6)
    ulp = np.exp2(e - 3.0)
    q = a / ulp
    n = np.floor(q)
    r = q - n
    up = (r > 0.5) | ((r == 0.5) & (np.mod(n, 2) == 1))
    val = np.minimum((n + up) * ulp, E4M3_MAX)
    # encode: subnormal m * 2^-9, else ((e + 7) << 3) | mantissa
    _, pv = np.frexp(val)
    ev = pv - 1
    normal = val >= 2.0 ** -6
    mant = np.where(normal, (val / np.exp2(np.where(normal, ev, 0)) - 1.0) * 8.0, 0.0)
    code = np.where(normal, ((ev + 7) << 3) + np.round(mant).astype(np.int64), np.round(val / 2.0 ** -9).astype(np.int64))
    code = np.where(np.isnan(x), NAN_CODE, sign | code)
    return code.astype(np.uint8)


def quantize_rows(a):
    """Per-row E4M3 quantization of an fp32 (or bf16-valued) matrix [R, K]:
    returns (codes uint8 [R, K], scales fp32 [R])."""
    a = np.asarray(a, dtype=np.float32)
    R = a.shape[0]
    codes = np.zeros(a.shape, dtype=np.uint8)
    scales = np.ones(R, dtype=np.float32)
    for r in range(R):
        amax = np.float32(np.max(np.abs(a[r]))) if a.shape[1] else np.float32(0)
        if amax == 0:
            continue
        s = np.float32(amax / np.float32(E4M3_MAX))
        scales[r] = s
        codes[r] = e4m3_round((a[r] / s).astype(np.float32))
    return codes, scales


def dequantize_rows(codes, scales) -> np.ndarray:
    """Float64 values represented by (codes, per-row scales)."""
    return e4m3_decode(codes) * np.asarray(scales, dtype=np.float64)[:, None]


def draft_layer_fp8(x, Wq, w_scale):
    """Draft layer on FP8 weights: x fp32/bf16-valued [M, K] is quantized per
    token row, then y = s_x s_w (xq . Wq) in float64 [M, N] (before bf16)."""
    xq, sx = quantize_rows(x)
    acc = e4m3_decode(xq) @ e4m3_decode(Wq).T  # exact products, float64 sums
    return acc * np.asarray(sx, np.float64)[:, None] * np.asarray(w_scale, np.float64)[None, :]
