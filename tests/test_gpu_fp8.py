"""GPU parity of the FP8 draft pass (mlora_quantize_rows_fp8, mlora_linear_fp8)
with the oracle (oracle.fp8).

Codes and scales are decided in fp32 on both sides (IEEE division, round to
nearest even, saturation), so they must match bit for bit.  The layer output
is compared with the oracle's float64 value: the products of two E4M3 codes
are exact in fp32, the tensor cores add them in fp32, the epilogue multiplies
by the two scales and rounds to bf16.  Tolerance per entry:
|y - y_ref| <= 2^-8 |y_ref| + 2^-12 S, with S = s_x s_w sum_k |xq wq| (the
bf16 rounding is 2^-9 relative; fp32 sums of up to 27648 terms err by far less
than 2^-12 of the absolute sum).  The quality check against the bf16 layer is
the relative error of the whole output (the format's 3 mantissa bits: a few
percent).
"""
import numpy as np
import pytest
import torch

import workloads as WL
from oracle import fp8 as F
from oracle import layer as OL
from tests.gpu_util import dev, dev_bf16, needs_gpu

pytestmark = pytest.mark.gpu


def _bf16_rows(g, R, K, std=1.0):
    return WL._normal_bf16(g, (R, K), std)


def _f32(bits):
    return WL.bf16_to_f64(bits).astype(np.float32)


def _check_layer(y_gpu, xb, Wq, sw, rows=None, cols=None):
    x = _f32(xb)
    y_ref = F.draft_layer_fp8(x, Wq, sw)
    xq, sx = F.quantize_rows(x)
    S = (np.abs(F.e4m3_decode(xq)) @ np.abs(F.e4m3_decode(Wq)).T) * sx[:, None].astype(np.float64) \
        * np.asarray(sw, np.float64)[None, :]
    y = y_gpu.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        y = y[np.ix_(rows, cols)]
    err = np.abs(y - y_ref)
    assert np.all(err <= 2.0 ** -8 * np.abs(y_ref) + 2.0 ** -12 * S + 1e-30), float(np.max(err / (S + 1e-30)))
    return y_ref


@pytest.mark.parametrize("R,K", [(1, 16), (7, 272), (64, 5120), (3, 27648)])
def test_quantize_rows_bit_exact(R, K):
    ml = needs_gpu()
    g = np.random.default_rng(R * 1000 + K)
    a = _bf16_rows(g, R, K, 0.02)
    if R >= 3:
        a[1] = 0x8000  # a row of negative zeros: scale 1, +0 codes
        big = _f32(a[2:3]) * np.exp2(g.integers(-20, 6, (1, K))).astype(np.float32)  # wide dynamic range
        a[2] = WL.bf16_bits(big)[0]
    q, s = ml.quantize_rows_fp8(dev_bf16(a))
    q_ref, s_ref = F.quantize_rows(_f32(a))
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(q.cpu().numpy(), q_ref)


@pytest.mark.parametrize("M,N,K", [(1, 128, 16), (17, 1000, 272), (128, 384, 512), (256, 640, 1024), (64, 129, 4096)])
def test_linear_fp8_against_oracle(M, N, K):
    ml = needs_gpu()
    g = np.random.default_rng(M + N + K)
    Wb = _bf16_rows(g, N, K, 1.0 / np.sqrt(K))
    xb = _bf16_rows(g, M, K, 1.0)
    xb[0, : min(K, 8)] = 0  # some zeros
    W8, sw = ml.quantize_rows_fp8(dev_bf16(Wb))
    Wq, sw_ref = F.quantize_rows(_f32(Wb))
    assert np.array_equal(W8.cpu().numpy(), Wq) and np.array_equal(sw.cpu().numpy(), sw_ref)
    y = ml.linear_fp8(dev_bf16(xb), W8, sw)
    y_ref = _check_layer(y, xb, Wq, sw_ref)
    # quality against the bf16 layer (LoRA off): the E4M3 rounding of W and x
    exact, _ = OL.mlora_linear(WL.bf16_to_f64(xb), WL.bf16_to_f64(Wb), None, None, None, None, 0.0, OL.DRAFT)
    rel = np.linalg.norm(y_ref - exact) / np.linalg.norm(exact)
    assert rel < 0.06, rel


def test_zero_rows_and_prefetch_flag():
    ml = needs_gpu()
    g = np.random.default_rng(5)
    M, N, K = 40, 256, 384
    Wb = _bf16_rows(g, N, K, 0.05)
    Wb[3] = 0
    xb = _bf16_rows(g, M, K)
    xb[7] = 0
    W8, sw = ml.quantize_rows_fp8(dev_bf16(Wb))
    ws = ml.Workspace(ml.linear_fp8_workspace_bytes(M, N, K))
    y1 = ml.linear_fp8(dev_bf16(xb), W8, sw, ws=ws)
    y2 = ml.linear_fp8(dev_bf16(xb), W8, sw, flags=ml.PREFETCH_WEIGHTS, ws=ws)
    assert torch.equal(y1, y2) and ws.status() == 0
    yh = y1.float().cpu().numpy()
    assert not yh[7].any() and not yh[:, 3].any()
    _check_layer(y1, xb, F.quantize_rows(_f32(Wb))[0], F.quantize_rows(_f32(Wb))[1])


@pytest.mark.parametrize("proj", ["q_k_v", "o", "gate_up", "down"])
def test_full_size_32b_draft_sampled(proj):
    """The 32B block's draft projections at 128 rows: W generated on the
    device, every output checked on 24 sampled W rows (the oracle quantizes
    those rows itself; the GPU's codes for them must match bit for bit)."""
    ml = needs_gpu()
    N, K = {"q_k_v": (7168, 5120), "o": (5120, 5120), "gate_up": (55296, 5120), "down": (5120, 27648)}[proj]
    M = 128
    gen = torch.Generator(device="cuda")
    gen.manual_seed(N + K)
    W = (torch.randn((N, K), generator=gen, device="cuda") / np.sqrt(K)).to(torch.bfloat16)
    x = torch.randn((M, K), generator=gen, device="cuda").to(torch.bfloat16)
    W8, sw = ml.quantize_rows_fp8(W)
    y = ml.linear_fp8(x, W8, sw)
    cols = np.sort(np.random.default_rng(N).choice(N, 24, replace=False))
    cols[-1] = N - 1
    Wb = W[torch.from_numpy(cols).cuda()].view(torch.int16).cpu().numpy().view(np.uint16)
    xb = x.view(torch.int16).cpu().numpy().view(np.uint16)
    Wq, sw_ref = F.quantize_rows(_f32(Wb))
    assert np.array_equal(W8[torch.from_numpy(cols).cuda()].cpu().numpy(), Wq)
    assert np.array_equal(sw[torch.from_numpy(cols).cuda()].cpu().numpy(), sw_ref)
    _check_layer(y, xb, Wq, sw_ref, rows=np.arange(M), cols=cols)
    del W, W8
    torch.cuda.empty_cache()
