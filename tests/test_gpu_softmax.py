"""GPU parity of the softmax, the draft draw and the accept step on logits.

The kernels compute a probability as e^(z - m) R in fp32 (e^d = 2^(d log2 e)
by the ex2.approx instruction, R = 1/S rounded once per row); the oracle is
the float64 softmax.  Tolerance: per entry |p - p_ref| <= REL * p_ref with
REL = 1e-4, from the fp32 arithmetic: the rounding of z - m and of the
product with log2 e move the exponent by under |z - m| 2^-23 (under 5e-6
for the |z - m| <= 40 of these inputs), ex2.approx errs by about 2^-22
relative, the row sum (16 terms per lane, 5 tree levels inside a block, a
block's rescaling, then up to blocks / 32 terms per lane and 5 more levels)
errs by under 1e-5 relative for V up to 2^20, and the reciprocal and the
product add an ulp.

The draw and the accept decisions are integers decided by those fp32 values,
so they are compared with the oracle run on the float64 probabilities
rounded to fp32: every request on which the two disagree must lie inside
the rounding margin (an accept test with |u q - p| <= REL (p + q), or a draw
whose threshold T lies within the weights' largest possible shift of a
cumulative boundary), and disagreements must be rare.  (The margin is a
worst case that adds every entry's error in one direction; on a flat
128256-entry row most draws lie inside it, so it decides only which
disagreements are allowed, not which requests are compared.)
Inside the CUDA path the logits form must equal, bit for bit, the probability
form fed with the probabilities mlora_softmax writes (one formula for every
entry).
"""
import numpy as np
import pytest
import torch

import workloads as WL
from oracle import accept as OA
from oracle import softmax as OS
from tests.gpu_util import dev, needs_gpu

pytestmark = pytest.mark.gpu
REL = 1e-4


def _check_probs(p_gpu, z):
    p_ref = OS.softmax(np.asarray(z, np.float64))
    p = p_gpu.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(p - p_ref) <= REL * p_ref + 1e-30), float(np.max(np.abs(p - p_ref) / np.maximum(p_ref, 1e-30)))


def _draw_margin(w, U):
    """Distance from T = floor(U S / 2^32) to the nearest cumulative boundary."""
    S = int(w.sum(dtype=np.uint64))
    if S == 0:
        return np.inf
    T = (int(U) * S) >> 32
    c = np.cumsum(w.astype(np.float64))
    return float(np.min(np.abs(c - T)))


def _weights_shift(V, n_rows):
    # Q(p) = floor(p 2^40): each weight moves by at most REL p 2^40 + 1 per row read,
    # so a cumulative sum (and the total S, hence T) by at most REL 2^40 + V per row.
    return n_rows * (REL * 2.0 ** 40 + V)


@pytest.mark.parametrize("rows,V", [(1, 1), (3, 5), (8, 1000), (5, 4099), (16, 128256), (40, 128256)])
def test_softmax_matches_float64(rows, V):
    ml = needs_gpu()
    g = np.random.default_rng(rows + V)
    z = (g.standard_normal((rows, V)) * 3).astype(np.float32)
    if V > 3:
        z[0, 2] = -np.inf          # a masked token: probability exactly 0
        z[-1, 1] = np.float32(200.0)  # one logit that dominates its row
    p = ml.softmax(dev(z))
    assert p.cpu().numpy()[0, 2] == 0.0 if V > 3 else True
    _check_probs(p, z)
    assert torch.equal(p, ml.softmax(dev(z)))  # deterministic
    # A row's statistics do not depend on the other rows of the call (nor on
    # the grid that takes its chunks).
    assert torch.equal(p[-1:], ml.softmax(dev(z[-1:])))


@pytest.mark.parametrize("B,V", [(256, 128256), (9, 1000), (7, 4099), (3, 600000), (1, 1 << 24)])
def test_draft_sample_against_oracle(B, V):
    ml = needs_gpu()
    zq = WL.accept_logits(V, B, 1, seed=B)[1][:, 0].copy()
    u = np.random.default_rng(V).random(B, dtype=np.float32)
    u[0] = np.float32(0.0)
    tok, q = ml.draft_sample(dev(zq), dev(u))
    _check_probs(q, zq)
    assert torch.equal(q, ml.softmax(dev(zq)))  # the draw used the library's probabilities
    # On the kernel's own probabilities the draw is integer work: bit-exact.
    assert np.array_equal(tok.cpu().numpy(), OS.draft_sample(q.cpu().numpy(), u))
    # The same logits through a view 4 bytes off 16-byte alignment (the
    # kernels' scalar-load path) give the same probabilities and tokens.
    tok2, q2 = ml.draft_sample(_offset_copy(zq), dev(u))
    assert torch.equal(tok2, tok) and torch.equal(q2, q)
    assert torch.equal(ml.softmax(_offset_copy(zq)), q)
    q_ref32 = OS.softmax(zq.astype(np.float64)).astype(np.float32)
    tok_ref = OS.draft_sample(q_ref32, u)
    tok = tok.cpu().numpy()
    differ = [b for b in range(B) if tok[b] != tok_ref[b]]
    for b in differ:  # a disagreement is allowed only inside the rounding margin
        U = int(np.floor(np.float64(u[b]) * 2.0 ** 32))
        assert _draw_margin(OA.quantize(q_ref32[b]), U) <= 2 * _weights_shift(V, 1), b
    assert len(differ) <= max(1, B // 100), differ


def _offset_copy(a):
    flat = torch.empty(a.size + 1, dtype=torch.float32, device="cuda")
    view = flat[1:].view(a.shape)
    view.copy_(torch.from_numpy(np.ascontiguousarray(a)))
    return view


# (6000, 5, 5): 66000 statistics rows, more than one launch takes (65536), split
# inside the draft rows.
@pytest.mark.parametrize("B,k,V", [(64, 1, 128256), (32, 3, 128256), (16, 2, 4099), (8, 4, 1000), (3, 1, 5),
                                   (6000, 5, 5)])
def test_accept_on_logits(B, k, V):
    ml = needs_gpu()
    zp, zq, tok, u = WL.accept_logits(V, B, k, sigma=0.3, seed=V + k)
    u[::5, 0] = np.float32(0.999)  # some rejections at position 0
    # Inside the CUDA path: the logits form equals the probability form on mlora_softmax's output.
    for mk in (dev, _offset_copy):
        ws = ml.Workspace(ml.accept_workspace_bytes(B, k, V))
        out, acc = ml.verify_accept_logits(mk(zp), mk(zq), dev(tok), dev(u), ws=ws)
        st = ws.status()
        p_gpu, q_gpu = ml.softmax(dev(zp)), ml.softmax(dev(zq))
        ws2 = ml.Workspace(ml.accept_workspace_bytes(B, k, V))
        out2, acc2 = ml.verify_accept(p_gpu, q_gpu, dev(tok), dev(u), ws=ws2)
        assert torch.equal(out, out2) and torch.equal(acc, acc2) and st == ws2.status()
    out, acc = out.cpu().numpy(), acc.cpu().numpy()
    # Against the oracle on the float64 probabilities rounded to fp32.
    p32 = OS.softmax(zp.astype(np.float64)).astype(np.float32)
    q32 = OS.softmax(zq.astype(np.float64)).astype(np.float32)
    out_r, acc_r, _ = OA.verify_accept(p32, q32, tok, u)
    differ = [b for b in range(B) if acc[b] != acc_r[b] or not np.array_equal(out[b], out_r[b])]
    for b in differ:  # a disagreement is allowed only inside the rounding margin
        close = False
        for i in range(min(int(acc_r[b]) + 1, k)):
            x = int(tok[b, i])
            pi, qi = float(p32[b, i, x]), float(q32[b, i, x])
            close |= abs(float(u[b, i]) * qi - pi) <= REL * (pi + qi) + 1e-30
        n = int(acc_r[b])
        if n < k:
            w = np.maximum(OA.quantize(p32[b, n]).astype(np.int64) - OA.quantize(q32[b, n]).astype(np.int64), 0)
            shift = _weights_shift(V, 2)
        else:
            w = OA.quantize(p32[b, k]).astype(np.int64)
            shift = _weights_shift(V, 1)
        U = int(np.floor(np.float64(min(u[b, k], np.float32(1) - np.float32(2 ** -24))) * 2.0 ** 32))
        close |= _draw_margin(w.astype(np.uint64), U) <= 2 * shift
        assert close, b
    assert len(differ) <= max(1, B // 50), differ


def test_q40_matches_cuda_conversion_on_every_float():
    """The draw's Q(f) = floor(f 2^40), computed from the bits of f, equals
    CUDA's round-down conversion of the clamped f 2^40 on all 2^32 fp32 bit
    patterns (zeros, subnormals, values above 1, infinities and NaNs
    included)."""
    ml = needs_gpu()
    lib = ml.library()
    bad = torch.zeros(1, dtype=torch.int64, device="cuda")
    for first in (0, 1 << 31):
        assert lib.mlora_debug_q40_mismatches(first, 1 << 31, bad.data_ptr(), None) == 0
    torch.cuda.synchronize()
    assert int(bad.item()) == 0
    # The range check: first + count past 2^32 is refused.
    assert lib.mlora_debug_q40_mismatches(2, 0xFFFFFFFF, bad.data_ptr(), None) != 0


def _exp_max_rel(lib, lo, hi):
    """Largest relative difference between the kernels' e^d and CUDA's expf
    over every fp32 d in [lo, hi] (lo <= hi <= 0)."""
    import struct
    bits = lambda f: struct.unpack("<I", struct.pack("<f", f))[0]  # noqa: E731
    first, last = bits(float(hi)) if hi < 0 else 0x80000000, bits(float(lo))
    out = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert lib.mlora_debug_exp_max_rel_error(first, last - first + 1, out.data_ptr(), None) == 0
    if hi >= 0:  # d = +0 as well
        assert lib.mlora_debug_exp_max_rel_error(0, 1, out.data_ptr(), None) == 0
    torch.cuda.synchronize()
    return float(out.cpu().view(torch.float32).item())


def test_exp_against_cuda_expf():
    """e^d = 2^(d log2 e) by ex2.approx against CUDA's expf on every fp32 d in
    [-87, 0].  The error comes from rounding y = d log2 e (half an ulp of y:
    2^-18 for |y| < 128, 2^-19 for |y| < 64), from log2 e rounded to fp32
    (1.3e-8 relative, so |y| * 1.3e-8 absolute), each moving e^d by ln 2 times
    that, plus ex2.approx's and expf's own few-ulp errors: about 4.3e-6
    relative over the whole range and 2.2e-6 for |d| <= 40.  The limits
    below leave room for the two instructions' errors."""
    ml = needs_gpu()
    lib = ml.library()
    near = _exp_max_rel(lib, -40.0, 0.0)
    full = _exp_max_rel(lib, -87.0, 0.0)
    assert 0.0 < near <= 4e-6, near
    assert near <= full <= 8e-6, full
    bad = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert lib.mlora_debug_exp_max_rel_error(2, 0xFFFFFFFF, bad.data_ptr(), None) != 0


def test_draft_sample_uniform_edge_cases():
    """Uniforms outside [0, 1) are clamped as the accept step clamps them (NaN
    and negatives to 0, 1 and above to the largest float below 1) and raise
    MLORA_DEV_BAD_PROB; the tokens equal the oracle's on the kernel's own
    probabilities, including the draws at the two ends of the range."""
    ml = needs_gpu()
    V, B = 1000, 6
    zq = WL.accept_logits(V, B, 1, seed=5)[1][:, 0].copy()
    below_one = np.nextafter(np.float32(1), np.float32(0))
    u = np.array([np.nan, -1.0, 1.5, 1.0, below_one, 0.0], dtype=np.float32)
    ws = ml.Workspace(int(ml.library().mlora_draft_sample_workspace_bytes(B, V)))
    tok, q = ml.draft_sample(dev(zq), dev(u), ws=ws)
    assert ws.status() & ml.DEV_BAD_PROB
    assert np.array_equal(tok.cpu().numpy(), OS.draft_sample(q.cpu().numpy(), u))
    # u = 0 draws the first token with weight; the largest u the last one.
    w = OA.quantize(q.cpu().numpy())
    assert tok[5].item() == int(np.flatnonzero(w[5])[0])
    assert tok[4].item() == int(np.flatnonzero(w[4])[-1])
    # Only valid uniforms: no status bit.
    ws2 = ml.Workspace(int(ml.library().mlora_draft_sample_workspace_bytes(B, V)))
    ml.draft_sample(dev(zq), dev(np.full(B, 0.5, dtype=np.float32)), ws=ws2)
    assert ws2.status() == 0
