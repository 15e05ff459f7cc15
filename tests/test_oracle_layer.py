"""Pins for the float64 layer oracle against facts fixed outside the oracle.

Each pin is chosen so that a plausible slip in the oracle (a dropped scale,
a transposed A or B, a wrong rank slice, adapters swapped between rows, the
low-rank term applied in draft mode) fails at least one of them.
"""
import json
import os

import numpy as np
import pytest

from oracle import layer as OL
import workloads as WL

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _case(seed=0, M=11, K=24, N=20, n_ad=4, ranks=(1, 2, 3, 0), r_max=4, pad_nan=True):
    g = np.random.default_rng(seed)
    x = g.standard_normal((M, K))
    W = g.standard_normal((N, K))
    A = np.full((n_ad, r_max, K), np.nan if pad_nan else 0.0)
    B = np.full((n_ad, N, r_max), np.nan if pad_nan else 0.0)
    for a, r in enumerate(ranks):
        A[a, :r] = g.standard_normal((r, K))
        B[a, :, :r] = g.standard_normal((N, r))
    idx = g.integers(-1, n_ad, M).astype(np.int32)
    return x, W, A, B, np.asarray(ranks, np.int32), idx


def _brute(x, W, A, B, ranks, idx, scale, mode):
    """Pure-Python loops over the definition, for tiny sizes."""
    M, K = len(x), len(x[0])
    N = len(W)
    y = [[0.0] * N for _ in range(M)]
    for m in range(M):
        a = int(idx[m])
        for n in range(N):
            acc = 0.0
            for k in range(K):
                acc += float(W[n][k]) * float(x[m][k])
            if mode == OL.VERIFY and a >= 0 and int(ranks[a]) > 0:
                low = 0.0
                for j in range(int(ranks[a])):
                    t = 0.0
                    for k in range(K):
                        t += float(A[a][j][k]) * float(x[m][k])
                    low += float(B[a][n][j]) * t
                acc += scale * low
            y[m][n] = acc
    return np.asarray(y)


def test_hand_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "layer_hand_example.json")))
    args = [np.asarray(g[k], dtype=np.float64) for k in ("x", "W", "A_stack", "B_stack")]
    ranks = np.asarray(g["rank_of"], np.int32)
    idx = np.asarray(g["adapter_idx"], np.int32)
    yv, st = OL.mlora_linear(*args, ranks, idx, g["scale"], OL.VERIFY)
    yd, _ = OL.mlora_linear(*args, ranks, idx, g["scale"], OL.DRAFT)
    assert st == 0
    assert np.array_equal(yv, np.asarray(g["y_verify"], np.float64))
    assert np.array_equal(yd, np.asarray(g["y_draft"], np.float64))


@pytest.mark.parametrize("mode", [OL.DRAFT, OL.VERIFY])
def test_brute_force_tiny(mode):
    x, W, A, B, ranks, idx = _case(M=5, K=6, N=7, n_ad=3, ranks=(1, 3, 2))
    y, _ = OL.mlora_linear(x, W, A, B, ranks, idx, 1.75, mode)
    yb = _brute(x, W, A, B, ranks, idx, 1.75, mode)
    assert np.allclose(y, yb, rtol=1e-12, atol=1e-12)


def test_merged_weight_identity():
    """(W + s B_a A_a) x = W x + s B_a (A_a x): the merged-weight form of the
    "LoRA Inference" glossary (W = W0 + dW) gives the same output."""
    x, W, A, B, ranks, idx = _case(seed=3, ranks=(1, 2, 3, 4))
    s = 0.625
    y, _ = OL.mlora_linear(x, W, A, B, ranks, idx, s, OL.VERIFY)
    for m in range(x.shape[0]):
        a = int(idx[m])
        Wm = W.copy()
        if a >= 0:
            r = int(ranks[a])
            Wm = W + s * B[a][:, :r] @ A[a][:r, :]
        ref = Wm @ x[m]
        assert np.max(np.abs(y[m] - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


def test_zero_B_and_zero_A_reduce_to_base_gemm():
    x, W, A, B, ranks, idx = _case(seed=4, pad_nan=False, ranks=(2, 2, 3, 1))
    base = x @ W.T
    y0, _ = OL.mlora_linear(x, W, A, np.zeros_like(B), ranks, idx, 3.0, OL.VERIFY)
    assert np.array_equal(y0, base)
    y1, _ = OL.mlora_linear(x, W, np.zeros_like(A), B, ranks, idx, 3.0, OL.VERIFY)
    assert np.array_equal(y1, base)
    y2, _ = OL.mlora_linear(x, W, A, B, ranks, np.full_like(idx, -1), 3.0, OL.VERIFY)
    assert np.array_equal(y2, base)
    y3, _ = OL.mlora_linear(x, W, A, B, ranks, idx, 3.0, OL.DRAFT)
    assert np.array_equal(y3, base)
    # rank 0 adapters contribute nothing
    y4, _ = OL.mlora_linear(x, W, A, B, np.zeros_like(ranks), idx, 3.0, OL.VERIFY)
    assert np.array_equal(y4, base)


def test_scale_enters_linearly():
    x, W, A, B, ranks, idx = _case(seed=5, ranks=(1, 2, 3, 4))
    base = x @ W.T
    y1, _ = OL.mlora_linear(x, W, A, B, ranks, idx, 1.0, OL.VERIFY)
    y3, _ = OL.mlora_linear(x, W, A, B, ranks, idx, 3.0, OL.VERIFY)
    assert np.allclose(y3 - base, 3.0 * (y1 - base), rtol=1e-10, atol=1e-10)


def test_row_permutation_equivariance():
    x, W, A, B, ranks, idx = _case(seed=6, M=17)
    y, _ = OL.mlora_linear(x, W, A, B, ranks, idx, 2.0, OL.VERIFY)
    perm = np.random.default_rng(0).permutation(17)
    yp, _ = OL.mlora_linear(x[perm], W, A, B, ranks, idx[perm], 2.0, OL.VERIFY)
    assert np.allclose(yp, y[perm], rtol=1e-13, atol=1e-13)


def test_adapter_relabeling_invariance():
    x, W, A, B, ranks, idx = _case(seed=7, ranks=(1, 2, 3, 4))
    y, _ = OL.mlora_linear(x, W, A, B, ranks, idx, 2.0, OL.VERIFY)
    relabel = np.array([2, 0, 3, 1])          # old id -> new id
    inv = np.argsort(relabel)                 # new id -> old id
    idx2 = np.where(idx >= 0, relabel[np.maximum(idx, 0)], -1)
    y2, _ = OL.mlora_linear(x, W, A[inv], B[inv], ranks[inv], idx2, 2.0, OL.VERIFY)
    assert np.allclose(y2, y, rtol=1e-13, atol=1e-13)


def test_rank_padding_is_never_read():
    x, W, A, B, ranks, idx = _case(seed=8, pad_nan=True, ranks=(1, 2, 3, 0))
    y, st = OL.mlora_linear(x, W, A, B, ranks, idx, 2.0, OL.VERIFY)
    assert np.isfinite(y).all() and st == 0
    T, _ = OL.shrink(x, A, ranks, idx)
    assert np.isfinite(T).all()


def test_invalid_adapter_and_rank_flags():
    x, W, A, B, ranks, idx = _case(seed=9, pad_nan=False, ranks=(1, 2, 3, 4))
    bad = idx.copy()
    bad[0] = 7
    bad[1] = -5
    y, st = OL.mlora_linear(x, W, A, B, ranks, bad, 2.0, OL.VERIFY)
    assert st & OL.STATUS_BAD_ADAPTER
    assert np.allclose(y[:2], (x @ W.T)[:2], rtol=1e-14, atol=1e-14)
    r2 = ranks.copy()
    r2[1] = 99
    _, st2 = OL.mlora_linear(x, W, A, B, r2, idx, 2.0, OL.VERIFY)
    assert st2 & OL.STATUS_BAD_RANK


def test_plan_is_a_stable_sort():
    g = np.random.default_rng(10)
    for M, n_ad in [(1, 1), (16, 4), (128, 16), (512, 128), (37, 3)]:
        idx = g.integers(-1, n_ad, M).astype(np.int32)
        seg, perm, st = OL.plan_segments(idx, n_ad)
        bucket = np.where(idx < 0, n_ad, idx)
        assert np.array_equal(perm, np.argsort(bucket, kind="stable"))
        counts = np.bincount(bucket, minlength=n_ad + 1)
        assert np.array_equal(seg, np.concatenate([[0], np.cumsum(counts)]))
        assert st == 0


def test_shrink_matches_brute_force():
    x, W, A, B, ranks, idx = _case(seed=11, M=6, K=5, N=3, n_ad=3, ranks=(2, 1, 3))
    T, _ = OL.shrink(x, A, ranks, idx)
    for m in range(6):
        a = int(idx[m])
        for j in range(A.shape[1]):
            want = 0.0
            if a >= 0 and j < ranks[a]:
                want = sum(A[a, j, k] * x[m, k] for k in range(5))
            assert abs(T[m, j] - want) <= 1e-12


def test_entries_match_full_output():
    x, W, A, B, ranks, idx = _case(seed=12, M=9, K=16, N=12, ranks=(1, 2, 3, 4))
    y, _ = OL.mlora_linear(x, W, A, B, ranks, idx, 1.5, OL.VERIFY)
    g = np.random.default_rng(1)
    rows, cols = g.integers(0, 9, 40), g.integers(0, 12, 40)
    e = OL.mlora_linear_entries(rows, cols, x, W, A, B, ranks, idx, 1.5, OL.VERIFY)
    assert np.allclose(e, y[rows, cols], rtol=1e-13, atol=1e-13)


def test_exact_integer_case_is_exact():
    """Small integers: every intermediate and y are integers below 256, so the
    result is exact in float64, fp32 and bf16 alike."""
    g = np.random.default_rng(13)
    M, K, N, n_ad, r = 5, 8, 8, 3, 2
    x = g.integers(-2, 3, (M, K)).astype(np.float64)
    W = g.integers(-2, 3, (N, K)).astype(np.float64)
    A = g.integers(-1, 2, (n_ad, r, K)).astype(np.float64)
    B = g.integers(-1, 2, (n_ad, N, r)).astype(np.float64)
    idx = np.array([0, 2, -1, 1, 0], np.int32)
    y, _ = OL.mlora_linear(x, W, A, B, np.full(n_ad, r, np.int32), idx, 2.0, OL.VERIFY)
    assert np.array_equal(y, np.round(y)) and np.abs(y).max() <= 256
    yb = _brute(x, W, A, B, np.full(n_ad, r), idx, 2.0, OL.VERIFY)
    assert np.array_equal(y, yb)


def test_workload_shapes_and_bf16_inputs():
    cfg = WL.TINY
    W, A, B, ranks = WL.projection_weights(cfg, 0)
    assert W.shape == (512, 512) and A.shape == (4, 8, 512) and B.shape == (4, 512, 8)
    x = WL.activations(cfg, 0, "verify")
    idx = WL.row_adapters(cfg, "verify")
    assert x.shape == (16, 512) and idx.shape == (16,)
    assert np.array_equal(idx[0::2], idx[1::2])       # 2 rows per request
    Wf = WL.bf16_to_f64(W)
    assert abs(Wf.std() - 1 / np.sqrt(512)) < 0.01 / np.sqrt(512) * 10
    y, st = OL.mlora_linear(WL.bf16_to_f64(x), Wf, WL.bf16_to_f64(A), WL.bf16_to_f64(B), ranks, idx,
                            cfg.scale, OL.VERIFY)
    assert st == 0 and np.isfinite(y).all()
