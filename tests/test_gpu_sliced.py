"""GPU parity of the sliced layer call (projections that read the same rows,
one launch) against the float64 oracle applied slice by slice.

Each output slice s of y is, by definition, the single-projection layer with
slice s of W, its own A stack and its rows of B; the oracle is called per
slice and the tolerance is that of the single-projection tests.
"""
import numpy as np
import pytest
import torch

import workloads as WL
from oracle import layer as OL
from tests.gpu_util import dev, dev_bf16, host_bf16_to_f64, needs_gpu

pytestmark = pytest.mark.gpu
TOL = 1e-2


def _rel_err(y, y_ref):
    return float(np.max(np.abs(y - y_ref)) / max(np.max(np.abs(y_ref)), 1e-30))


def _sliced_case(seed, M, widths, K, n_ad, ranks, r_max, nan_pad=True, frac_none=0.1):
    g = np.random.default_rng(seed)
    N = sum(widths)
    S = len(widths)
    x = WL.bf16_bits(g.standard_normal((M, K)).astype(np.float32))
    W = WL.bf16_bits((g.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32))
    A = np.full((S, n_ad, r_max, K), 0x7FC0 if nan_pad else 0, np.uint16)
    B = np.full((n_ad, N, r_max), 0x7FC0 if nan_pad else 0, np.uint16)
    for a, r in enumerate(ranks):
        for s in range(S):
            A[s, a, :r] = WL.bf16_bits((g.standard_normal((r, K)) / np.sqrt(K)).astype(np.float32))
        B[a, :, :r] = WL.bf16_bits((g.standard_normal((N, r)) / np.sqrt(max(r, 1))).astype(np.float32))
    idx = g.integers(0, n_ad, M).astype(np.int32)
    idx[g.random(M) < frac_none] = -1
    ends = list(np.cumsum(widths))
    return x, W, A, B, np.asarray(ranks, np.int32), idx, ends


def _oracle_sliced(x, W, A, B, ranks, idx, ends, scale, mode):
    f = WL.bf16_to_f64
    parts = []
    n0 = 0
    for s, n1 in enumerate(ends):
        y, _ = OL.mlora_linear(f(x), f(W[n0:n1]), f(A[s]), f(B[:, n0:n1]), ranks, idx, scale, mode)
        parts.append(y)
        n0 = n1
    return np.concatenate(parts, axis=1)


def _run_sliced(ml, x, W, A, B, ranks, idx, ends, scale, mode, ws=None, seg=None):
    return ml.linear_sliced(dev_bf16(x), dev_bf16(W), ends, dev_bf16(A), dev_bf16(B), dev(ranks), dev(idx), scale,
                            mode, ws=ws, seg_offsets_ptr=seg)


@pytest.mark.parametrize("M,widths,K,n_ad,ranks", [
    # stream-K or cluster kernel, up to 256 rows
    (16, (256, 128, 130), 2048, 4, (8, 16, 24, 0)),
    (128, (512, 128, 128), 4096, 16, (16,) * 16),
    # more expand blocks than k-blocks
    (40, (128, 200), 256, 6, (8, 16, 32, 64, 24, 40)),
    # more than 256 rows: cluster kernel, two MMAs per k-step
    (300, (384, 256), 512, 5, (64, 8, 33, 17, 1)),
    (640, (256, 512, 128), 1024, 24, tuple([8, 16, 32, 64, 48, 24] * 4)),
    # four slices
    (64, (128, 128, 256, 72), 1024, 3, (16, 32, 8)),
])
def test_sliced_matches_oracle_per_slice(M, widths, K, n_ad, ranks):
    ml = needs_gpu()
    x, W, A, B, rk, idx, ends = _sliced_case(M + K, M, widths, K, n_ad, ranks, r_max=64)
    N = ends[-1]
    ws = ml.Workspace(ml.linear_sliced_workspace_bytes(M, N, K, n_ad, len(ends)))
    for mode in (OL.DRAFT, OL.VERIFY):
        y_ref = _oracle_sliced(x, W, A, B, rk, idx, ends, 2.0, mode)
        y = _run_sliced(ml, x, W, A, B, rk, idx, ends, 2.0, mode, ws=ws)
        assert ws.status() == 0
        assert _rel_err(host_bf16_to_f64(y), y_ref) <= TOL, (M, widths, mode)


def test_one_slice_is_mlora_linear_bitwise():
    ml = needs_gpu()
    x, W, A, B, rk, idx, ends = _sliced_case(3, 96, (1024,), 2048, 8, (8, 16, 32, 64) * 2, r_max=64)
    for mode in (ml.DRAFT, ml.VERIFY):
        y1 = _run_sliced(ml, x, W, A, B, rk, idx, ends, 2.0, mode)
        y2 = ml.linear(dev_bf16(x), dev_bf16(W), dev_bf16(A[0]), dev_bf16(B), dev(rk), dev(idx), 2.0, mode)
        assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_windows_are_rewritten_for_every_plan():
    """The shrink writes every token window whole (member entries and zeros),
    so a second plan with other adapter rows on the same workspace sees none
    of the first plan's entries."""
    ml = needs_gpu()
    M, K, n_ad = 64, 2048, 8
    x, W, A, B, rk, idx1, ends = _sliced_case(11, M, (256, 128), K, n_ad, (16, 8, 24, 16, 32, 8, 16, 16), r_max=32,
                                              frac_none=0.0)
    idx2 = np.random.default_rng(12).permutation(idx1).astype(np.int32)
    idx2[::5] = -1
    ws = ml.Workspace(ml.linear_sliced_workspace_bytes(M, ends[-1], K, n_ad, 2))
    for idx in (idx1, idx2, idx1):
        seg, _ = ml.plan_segments(dev(idx), dev(rk), n_ad, 32, ws)
        y_ref = _oracle_sliced(x, W, A, B, rk, idx, ends, 2.0, OL.VERIFY)
        y = _run_sliced(ml, x, W, A, B, rk, idx, ends, 2.0, ml.VERIFY, ws=ws, seg=seg)
        assert _rel_err(host_bf16_to_f64(y), y_ref) <= TOL
    assert ws.status() == 0


@pytest.mark.parametrize("cfg,k", [(WL.LLAMA8B_R16, 1), (WL.LLAMA8B_HET, 1), (WL.QWEN32B_R16, 1), (WL.QWEN32B_R16, 2),
                                   (WL.QWEN32B_R16, 4)], ids=lambda v: getattr(v, "name", f"k={v}"))
def test_fused_groups_full_size_sampled(cfg, k):
    """The decode-step grouping (q|k|v, o, gate|up, down) at full size, for
    every layer workload and draft length: 512 sampled outputs per call
    against the oracle, one output at a time."""
    ml = needs_gpu()
    ranks = WL.adapter_ranks(cfg)
    f = WL.bf16_to_f64
    for group in WL.input_groups(cfg):
        Ws, As, Bs = [], [], []
        for p in group:
            W, A, B, _ = WL.projection_weights(cfg, p)
            Ws.append(W)
            As.append(A)
            Bs.append(B)
        W = np.concatenate(Ws, axis=0)
        A = np.stack(As)
        B = np.concatenate(Bs, axis=1)
        ends = list(np.cumsum([w.shape[0] for w in Ws]))
        N, K = W.shape
        for mode, name in ((OL.DRAFT, "draft"), (OL.VERIFY, "verify")):
            x = WL.activations(cfg, group[0], name, k=k)
            idx = WL.row_adapters(cfg, name, k=k)
            M = x.shape[0]
            ws = ml.Workspace(ml.linear_sliced_workspace_bytes(M, N, K, cfg.n_adapters, len(group)))
            y = host_bf16_to_f64(ml.linear_sliced(dev_bf16(x), dev_bf16(W), ends, dev_bf16(A), dev_bf16(B),
                                                  dev(ranks), dev(idx), cfg.scale, mode, ws=ws))
            assert ws.status() == 0 and np.isfinite(y).all()
            g = np.random.default_rng(group[0])
            rows, cols = g.integers(0, M, 512), g.integers(0, N, 512)
            got = y[rows, cols]
            want = np.empty(512)
            n0 = 0
            for s, n1 in enumerate(ends):
                sel = (cols >= n0) & (cols < n1)
                if sel.any():
                    want[sel] = OL.mlora_linear_entries(rows[sel], cols[sel] - n0, f(x), f(Ws[s]), f(As[s]),
                                                        f(Bs[s]), ranks, idx, cfg.scale, mode)
                n0 = n1
            assert np.max(np.abs(got - want)) <= TOL * max(np.max(np.abs(want)), 1e-30), (cfg.name, group, name)


def test_gemm_kernel_query():
    """mlora_linear_gemm_kernel names one of the two GEMM kernels for valid
    shapes and refuses invalid ones; on a 152-SM GB300 draft calls (LoRA
    off) take the stream-K kernel up to its 1024 rows; verify calls take the
    cluster kernel for one wave that fills 80% of the SMs (70% past 256
    rows)."""
    ml = needs_gpu()
    for M, N, K in [(64, 6144, 4096), (64, 4096, 4096), (64, 28672, 4096), (64, 4096, 14336), (700, 512, 512)]:
        for mode in (ml.DRAFT, ml.VERIFY):
            assert ml.gemm_kernel_name(M, N, K, 16, 16, mode) in ("gemm_kernel", "gemm_sk_kernel")
    with pytest.raises(ValueError):
        ml.gemm_kernel_name(64, 4096, 4097, 16, 16, ml.DRAFT)
    assert ml.gemm_kernel_name(1100, 512, 512, 16, 16, ml.DRAFT) == "gemm_kernel"  # past the stream-K kernel's 1024 rows
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        # 640 verify rows (the 32B block at k = 4): only q|k|v has one well-filled cluster wave
        assert ml.gemm_kernel_name(640, 55296, 5120, 64, 16, ml.VERIFY) == "gemm_sk_kernel"
        assert ml.gemm_kernel_name(640, 5120, 5120, 64, 16, ml.VERIFY) == "gemm_sk_kernel"
        assert ml.gemm_kernel_name(640, 5120, 27648, 64, 16, ml.VERIFY) == "gemm_sk_kernel"
        assert ml.gemm_kernel_name(640, 7168, 5120, 64, 16, ml.VERIFY) == "gemm_kernel"  # one wave, 74% full
        assert ml.gemm_kernel_name(384, 7168, 5120, 64, 16, ml.VERIFY) == "gemm_sk_kernel"  # 257..384 rows
        assert ml.gemm_kernel_name(64, 4096, 4096, 16, 16, ml.DRAFT) == "gemm_sk_kernel"
        assert ml.gemm_kernel_name(64, 4096, 14336, 16, 16, ml.DRAFT) == "gemm_sk_kernel"
        assert ml.gemm_kernel_name(64, 28672, 4096, 16, 16, ml.DRAFT) == "gemm_sk_kernel"
        assert ml.gemm_kernel_name(128, 6144, 4096, 16, 16, ml.VERIFY) == "gemm_sk_kernel"
