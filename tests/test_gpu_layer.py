"""GPU parity of the multi-LoRA layer (steps a1-a4) against the float64 oracle.

Tolerance: max |y - y_ref| <= 1e-2 * max |y_ref| per call (bf16 inputs, fp32
accumulation, one bf16 rounding of the output).  Integer work (the plan) and
the small-integer case are compared bit for bit.
"""
import ctypes

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


def _random_case(seed, M, N, K, n_ad, ranks, r_max, nan_pad=True, frac_none=0.1):
    g = np.random.default_rng(seed)
    x = WL.bf16_bits(g.standard_normal((M, K)).astype(np.float32))
    W = WL.bf16_bits((g.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32))
    A = np.full((n_ad, r_max, K), 0x7FC0 if nan_pad else 0, np.uint16)
    B = np.full((n_ad, N, r_max), 0x7FC0 if nan_pad else 0, np.uint16)
    for a, r in enumerate(ranks):
        A[a, :r] = WL.bf16_bits((g.standard_normal((r, K)) / np.sqrt(K)).astype(np.float32))
        B[a, :, :r] = WL.bf16_bits((g.standard_normal((N, r)) / np.sqrt(max(r, 1))).astype(np.float32))
    idx = g.integers(0, n_ad, M).astype(np.int32)
    idx[g.random(M) < frac_none] = -1
    return x, W, A, B, np.asarray(ranks, np.int32), idx


def _oracle(x, W, A, B, ranks, idx, scale, mode):
    f = WL.bf16_to_f64
    return OL.mlora_linear(f(x), f(W), f(A), f(B), ranks, idx, scale, mode)


def _run(ml, x, W, A, B, ranks, idx, scale, mode, ws=None):
    return ml.linear(dev_bf16(x), dev_bf16(W), dev_bf16(A), dev_bf16(B), dev(ranks), dev(idx), scale, mode, ws=ws)


def test_exact_small_integers_bitwise():
    ml = needs_gpu()
    g = np.random.default_rng(13)
    for (M, K, N, r) in [(5, 8, 8, 2), (19, 16, 24, 2), (33, 72, 130, 1)]:
        n_ad, r_max = 3, 8
        x = g.integers(-2, 3, (M, K)).astype(np.float32)
        W = g.integers(-2, 3, (N, K)).astype(np.float32)
        A = np.zeros((n_ad, r_max, K), np.float32)
        B = np.zeros((n_ad, N, r_max), np.float32)
        A[:, :r] = g.integers(-1, 2, (n_ad, r, K))
        B[:, :, :r] = g.integers(-1, 2, (n_ad, N, r))
        idx = g.integers(-1, n_ad, M).astype(np.int32)
        ranks = np.full(n_ad, r, np.int32)
        xb, Wb, Ab, Bb = (WL.bf16_bits(v) for v in (x, W, A, B))
        for mode in (OL.DRAFT, OL.VERIFY):
            y_ref, _ = _oracle(xb, Wb, Ab, Bb, ranks, idx, 2.0, mode)
            if np.abs(y_ref).max() > 256:
                continue
            y = host_bf16_to_f64(_run(ml, xb, Wb, Ab, Bb, ranks, idx, 2.0, mode))
            assert np.array_equal(y, y_ref), (M, K, N, mode)


def test_tiny_workload_both_modes():
    ml = needs_gpu()
    cfg = WL.TINY
    W, A, B, ranks = WL.projection_weights(cfg, 0)
    for mode, name in ((OL.DRAFT, "draft"), (OL.VERIFY, "verify")):
        x = WL.activations(cfg, 0, name)
        idx = WL.row_adapters(cfg, name)
        y_ref, _ = _oracle(x, W, A, B, ranks, idx, cfg.scale, mode)
        y = host_bf16_to_f64(_run(ml, x, W, A, B, ranks, idx, cfg.scale, mode))
        assert _rel_err(y, y_ref) <= TOL


@pytest.mark.parametrize("M,N,K,n_ad,ranks", [
    (1, 8, 8, 1, (8,)),
    (5, 130, 72, 3, (8, 0, 16)),
    (17, 200, 200, 4, (8, 16, 24, 64)),
    (100, 1000, 520, 8, (8, 16, 32, 64, 8, 16, 32, 64)),
    (257, 384, 1024, 5, (64, 8, 33, 17, 1)),
    (513, 256, 256, 6, (16,) * 6),
    (640, 1024, 384, 64, tuple([8, 16, 32, 64] * 16)),
    (700, 136, 128, 3, (8, 8, 8)),
])
def test_ragged_shapes_against_oracle(M, N, K, n_ad, ranks):
    ml = needs_gpu()
    x, W, A, B, rk, idx = _random_case(M * 7 + N, M, N, K, n_ad, ranks, r_max=64)
    for mode in (OL.DRAFT, OL.VERIFY):
        y_ref, _ = _oracle(x, W, A, B, rk, idx, 2.0, mode)
        ws = ml.Workspace(ml.linear_workspace_bytes(M, N, K, n_ad))
        y = _run(ml, x, W, A, B, rk, idx, 2.0, mode, ws=ws)
        assert ws.status() == 0
        assert _rel_err(host_bf16_to_f64(y), y_ref) <= TOL, (M, N, K, mode)


@pytest.mark.parametrize("M,N,K,n_ad,ranks", [
    (16, 256, 2048, 4, (8, 16, 24, 0)),    # ranks inside a 16-wide block: B columns zeroed before the MMA
    (64, 384, 4096, 4, (16, 32, 48, 64)),  # multiples of 16: padding never inside a block
    (128, 1024, 4096, 16, (16,) * 15 + (40,)),
    (128, 1024, 1024, 32, (16,) * 32),     # 32 blocks against a 1024-deep K loop
])
def test_nan_rank_padding_in_expand_shapes(M, N, K, n_ad, ranks):
    """NaN in every padding entry of A and B past each adapter's rank never
    reaches y."""
    ml = needs_gpu()
    x, W, A, B, rk, idx = _random_case(M + N + K, M, N, K, n_ad, ranks, r_max=64, nan_pad=True)
    y_ref, _ = _oracle(x, W, A, B, rk, idx, 2.0, OL.VERIFY)
    ws = ml.Workspace(ml.linear_workspace_bytes(M, N, K, n_ad))
    y = host_bf16_to_f64(_run(ml, x, W, A, B, rk, idx, 2.0, OL.VERIFY, ws=ws))
    assert ws.status() == 0 and np.isfinite(y).all()
    assert _rel_err(y, y_ref) <= TOL


def _zipf_idx(seed, M, n_ad, s=1.1):
    g = np.random.default_rng(seed)
    w = np.arange(1, n_ad + 1, dtype=np.float64) ** -s
    return g.choice(n_ad, M, p=w / w.sum()).astype(np.int32)


@pytest.mark.parametrize("M,N,K,n_ad,ranks,zipf", [
    # more than 256 rows: stream-K over token groups of at most 256 rows, sorted rows and token windows
    (384, 1024, 1024, 16, (8, 16, 32, 64) * 4, False),            # two groups of 192
    (512, 640, 2048, 128, tuple([8, 16, 32, 64] * 32), True),    # heterogeneous ranks, Zipf: large and single rows
    (640, 768, 1536, 64, (16,) * 64, False),                      # three groups of 224
    (1000, 256, 512, 40, tuple([8, 24, 40, 56, 64] * 8), True),   # four groups; windows crossing group boundaries
    # more than 256 rows in one well-filled cluster wave: cluster kernel, two MMAs per k-step, 320-row groups
    (640, 7168, 512, 64, (16,) * 64, False),
    # stream-K verify (at most 256 rows) with hundreds of expand blocks and ranks inside 16-wide blocks
    (256, 6144, 1024, 128, (64,) * 128, False),
    (200, 640, 2048, 64, (8, 24, 40, 56) * 16, True),
    (48, 1280, 4096, 300, tuple([1, 9, 17, 33, 63] * 60), False),
])
def test_windowed_expand_against_oracle(M, N, K, n_ad, ranks, zipf):
    """The tensor-core expand over each adapter's token window, with NaN in
    every padding entry of A and B past each adapter's rank."""
    ml = needs_gpu()
    x, W, A, B, rk, idx = _random_case(M + 3 * N + K, M, N, K, n_ad, ranks, r_max=64, nan_pad=True)
    if zipf:
        idx = _zipf_idx(M + n_ad, M, n_ad)
        idx[::11] = -1
    ws = ml.Workspace(ml.linear_workspace_bytes(M, N, K, n_ad))
    y_ref, _ = _oracle(x, W, A, B, rk, idx, 2.0, OL.VERIFY)
    y = host_bf16_to_f64(_run(ml, x, W, A, B, rk, idx, 2.0, OL.VERIFY, ws=ws))
    assert ws.status() == 0 and np.isfinite(y).all()
    assert _rel_err(y, y_ref) <= TOL, (M, N, K, n_ad, ml.gemm_kernel_name(M, N, K, n_ad, 64, ml.VERIFY))
    # every output row is written (rows come back through the permutation)
    yd = host_bf16_to_f64(_run(ml, x, W, A, B, rk, idx, 2.0, OL.DRAFT, ws=ws))
    y_ref_d, _ = _oracle(x, W, A, B, rk, idx, 2.0, OL.DRAFT)
    assert _rel_err(yd, y_ref_d) <= TOL


def test_stream_k_flag_wait_gives_up_and_workspace_recovers():
    """The stream-K GEMM's cross-CTA wait, made to run out on purpose: with
    the test hook the tile owners wait 2 microseconds on flag words nothing
    sets, give up, finish their tiles without the partial sums and raise the
    timeout bit; the call returns and the context stays usable.  After
    mlora_workspace_init the next call is back to oracle parity."""
    ml = needs_gpu()
    lib = ml.library()
    M, N, K = 64, 6144, 4096
    if ml.gemm_kernel_name(M, N, K, 4, 16, ml.DRAFT) != "gemm_sk_kernel":
        pytest.skip("this device runs the cluster kernel for the shape")
    x, W, A, B, rk, idx = _random_case(21, M, N, K, 4, (16, 16, 8, 12), r_max=16, nan_pad=False)
    ws = ml.Workspace(ml.linear_workspace_bytes(M, N, K, 4))
    lib.mlora_debug_set_flag_wait_ns(2000)
    try:
        _run(ml, x, W, A, B, rk, idx, 2.0, OL.DRAFT, ws=ws)
    finally:
        lib.mlora_debug_set_flag_wait_ns(0)
    bits = ctypes.c_uint32(0)
    st = lib.mlora_read_device_status(ws.ptr, ctypes.byref(bits), 1, torch.cuda.current_stream().cuda_stream)
    assert st == 6 and bits.value & ml.DEV_TIMEOUT  # MLORA_ERR_TIMEOUT
    assert lib.mlora_workspace_init(ws.ptr, ws.nbytes, torch.cuda.current_stream().cuda_stream) == 0
    y_ref, _ = _oracle(x, W, A, B, rk, idx, 2.0, OL.DRAFT)
    for mode in (OL.DRAFT, OL.VERIFY):
        y_ref, _ = _oracle(x, W, A, B, rk, idx, 2.0, mode)
        y = host_bf16_to_f64(_run(ml, x, W, A, B, rk, idx, 2.0, mode, ws=ws))
        assert ws.status() == 0
        assert _rel_err(y, y_ref) <= TOL


@pytest.mark.parametrize("M,N,K", [
    (64, 1024, 8192),    # cluster split-K over 16 CTAs
    (128, 4096, 4096),   # cluster split-K over 4 CTAs, one full wave
    (200, 640, 2048),    # stream-K, every tile split 4 ways
    (64, 6144, 4096),    # stream-K, the fused q|k|v shape
    (128, 14336, 4096),  # stream-K, the gate shape in verify mode
    (16, 28672, 4096),   # stream-K, the fused gate|up shape, few rows
    (1, 8, 512),         # stream-K, a single CTA
    (640, 640, 1024),    # stream-K, three token groups of 224 rows
    (384, 384, 2048),    # stream-K, two token groups of 192 rows
    (1024, 256, 512),    # stream-K, four token groups of 256 rows
])
def test_split_tiles_oracle_and_determinism(M, N, K):
    """Shapes whose tiles are shared by several CTAs, through both GEMM
    kernels: oracle parity, identical bits on repeated calls, and consecutive
    calls on one workspace (stream-K consumes the partial-sum flags it sets)."""
    ml = needs_gpu()
    x, W, A, B, rk, idx = _random_case(M + N + K, M, N, K, 4, (16, 16, 8, 12), r_max=16, nan_pad=True)
    ws = ml.Workspace(ml.linear_workspace_bytes(M, N, K, 4))
    for mode in (OL.DRAFT, OL.VERIFY):
        y_ref, _ = _oracle(x, W, A, B, rk, idx, 2.0, mode)
        ys = [_run(ml, x, W, A, B, rk, idx, 2.0, mode, ws=ws) for _ in range(3)]
        assert ws.status() == 0
        assert _rel_err(host_bf16_to_f64(ys[0]), y_ref) <= TOL, (M, N, K, mode)
        for y in ys[1:]:
            assert torch.equal(y.view(torch.int16), ys[0].view(torch.int16))


def test_plan_is_bit_exact():
    ml = needs_gpu()
    g = np.random.default_rng(2)
    for M, n_ad in [(1, 1), (16, 4), (128, 16), (512, 128), (640, 64), (3000, 4096), (5, 3)]:
        idx = g.integers(-1, n_ad, M).astype(np.int32)
        ranks = g.choice([0, 8, 16, 32, 64], n_ad).astype(np.int32)
        seg_ref, perm_ref, _ = OL.plan_segments(idx, n_ad)
        ws = ml.Workspace(ml.linear_workspace_bytes(M, 128, 64, n_ad))
        seg_p, perm_p = ml.plan_segments(dev(idx), dev(ranks), n_ad, 64, ws)
        seg = ws.view_int32(seg_p, n_ad + 2).cpu().numpy()
        perm = ws.view_int32(perm_p, M).cpu().numpy()
        assert np.array_equal(seg, seg_ref) and np.array_equal(perm, perm_ref), (M, n_ad)
        assert ws.status() == 0


def test_shrink_against_oracle():
    ml = needs_gpu()
    for (M, K, n_ad, ranks, zipf) in [(16, 512, 4, (8, 8, 8, 8), False),
                                      (512, 4096, 8, (8, 16, 32, 64, 1, 9, 63, 0), False),
                                      (37, 14336, 3, (16, 16, 16), False),
                                      (512, 14336, 128, _het_ranks(128, 3), True)]:
        x, W, A, B, rk, idx = _random_case(K + M, M, 8, K, n_ad, ranks, r_max=64)
        if zipf:  # heterogeneous ranks under Zipf(1.1): one segment of 100+ rows at rank 64, many singletons
            idx = _zipf_idx(M + n_ad, M, n_ad)
        T_ref, _ = OL.shrink(WL.bf16_to_f64(x), WL.bf16_to_f64(A), rk, idx)
        ws = ml.Workspace(ml.linear_workspace_bytes(M, 8, K, n_ad))
        seg_p, _ = ml.plan_segments(dev(idx), dev(rk), n_ad, 64, ws)
        T = ml.shrink(dev_bf16(x), dev_bf16(A), seg_p, ws).cpu().numpy().astype(np.float64)
        assert np.isfinite(T).all()
        assert np.max(np.abs(T - T_ref)) <= 1e-4 * max(np.max(np.abs(T_ref)), 1e-30)


def _het_ranks(n_ad, seed):
    rk = np.random.default_rng(seed).choice([8, 16, 32, 64], n_ad)
    rk[0] = 64  # the most popular adapter under Zipf: a segment of 100+ rows at rank 64
    return tuple(int(r) for r in rk)


@pytest.mark.parametrize("path", ["warp", "tensor"])
@pytest.mark.parametrize("M,K,n_ad,ranks,zipf", [
    (512, 14336, 128, _het_ranks(128, 3), True),  # 8B-shaped down projection, heterogeneous ranks, Zipf(1.1)
    (640, 5120, 64, (16,) * 64, False),           # 32B-shaped q|k|v input, draft length 4
    (300, 1024, 5, (64, 8, 33, 17, 1), False),    # ranks inside 16-wide blocks, segments of ~60 rows
    (1000, 512, 3, (64, 64, 16), False),          # segments of 300+ rows: windows wider than one MMA tile
    (7, 64, 3, (8, 16, 8), False),                # one k-block: no split of K
    (96, 2048, 40, tuple([1, 9, 17, 33, 63] * 8), True),
])
def test_lora_term_alone_both_shrink_paths(M, K, n_ad, ranks, zipf, path):
    """W = 0: the output is scale * B_a (A_a x) alone, so the low-rank operand
    (the shrink) is checked against the oracle at full relative weight, with
    NaN in every padding entry of A and B past each adapter's rank; both
    kernels that can write it (warp items, tensor-core tiles)."""
    ml = needs_gpu()
    N = 256
    x, W, A, B, rk, idx = _random_case(M + K + n_ad, M, N, K, n_ad, ranks, r_max=64, nan_pad=True)
    W[:] = 0
    if zipf:
        idx = _zipf_idx(M + n_ad, M, n_ad)
        idx[::13] = -1
    y_ref, _ = _oracle(x, W, A, B, rk, idx, 2.0, OL.VERIFY)
    ws = ml.Workspace(ml.linear_workspace_bytes(M, N, K, n_ad))
    ml.set_shrink_path(ml.SHRINK_WARP if path == "warp" else ml.SHRINK_TENSOR)
    try:
        y1 = _run(ml, x, W, A, B, rk, idx, 2.0, OL.VERIFY, ws=ws)
        y2 = _run(ml, x, W, A, B, rk, idx, 2.0, OL.VERIFY, ws=ws)
    finally:
        ml.set_shrink_path(ml.SHRINK_AUTO)
    assert ws.status() == 0
    y = host_bf16_to_f64(y1)
    assert np.isfinite(y).all() and np.abs(y_ref).max() > 0
    assert _rel_err(y, y_ref) <= TOL, (M, K, n_ad, path)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))  # deterministic


def test_set_shrink_path_rejects_unknown_values():
    ml = needs_gpu()
    with pytest.raises(ml.MLoraError):
        ml.set_shrink_path(3)
    ml.set_shrink_path(ml.SHRINK_AUTO)


def test_zero_B_verify_equals_draft_bitwise():
    ml = needs_gpu()
    x, W, A, B, rk, idx = _random_case(5, 128, 1024, 4096, 16, (16,) * 16, r_max=16, nan_pad=False)
    B[:] = 0
    yv = _run(ml, x, W, A, B, rk, idx, 2.0, OL.VERIFY)
    yd = _run(ml, x, W, A, B, rk, idx, 2.0, OL.DRAFT)
    assert torch.equal(yv.view(torch.int16), yd.view(torch.int16))


def test_row_permutation_and_determinism():
    ml = needs_gpu()
    x, W, A, B, rk, idx = _random_case(6, 96, 640, 1536, 8, (8, 16, 32, 64) * 2, r_max=64)
    y1 = _run(ml, x, W, A, B, rk, idx, 2.0, OL.VERIFY)
    y2 = _run(ml, x, W, A, B, rk, idx, 2.0, OL.VERIFY)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    perm = np.random.default_rng(1).permutation(96)
    yp = _run(ml, x[perm], W, A, B, rk, idx[perm], 2.0, OL.VERIFY)
    assert torch.equal(yp.view(torch.int16), y1[torch.from_numpy(perm).cuda()].view(torch.int16))


def test_adapter_relabeling_is_bitwise_invariant():
    ml = needs_gpu()
    x, W, A, B, rk, idx = _random_case(7, 64, 512, 512, 6, (8, 16, 32, 64, 24, 40), r_max=64, frac_none=0.0)
    y1 = _run(ml, x, W, A, B, rk, idx, 2.0, OL.VERIFY)
    relabel = np.array([3, 5, 0, 1, 4, 2])
    inv = np.argsort(relabel)
    y2 = _run(ml, x, W, A[inv].copy(), B[inv].copy(), rk[inv].copy(), relabel[idx].astype(np.int32), 2.0, OL.VERIFY)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_invalid_adapter_and_rank_raise_status():
    ml = needs_gpu()
    x, W, A, B, rk, idx = _random_case(8, 32, 256, 128, 4, (8, 8, 8, 8), r_max=8, nan_pad=False, frac_none=0.0)
    bad = idx.copy()
    bad[3] = 9
    bad[4] = -7
    y_ref, st_ref = _oracle(x, W, A, B, rk, bad, 2.0, OL.VERIFY)
    ws = ml.Workspace(ml.linear_workspace_bytes(32, 256, 128, 4))
    y = _run(ml, x, W, A, B, rk, bad, 2.0, OL.VERIFY, ws=ws)
    assert ws.status() == st_ref == ml.DEV_BAD_ADAPTER
    assert _rel_err(host_bf16_to_f64(y), y_ref) <= TOL
    rk2 = rk.copy()
    rk2[1] = 65
    y_ref, st_ref = _oracle(x, W, A, B, rk2, idx, 2.0, OL.VERIFY)
    y = _run(ml, x, W, A, B, rk2, idx, 2.0, OL.VERIFY, ws=ws)
    assert ws.status() == st_ref == ml.DEV_BAD_RANK
    assert _rel_err(host_bf16_to_f64(y), y_ref) <= TOL


def test_one_workspace_and_one_plan_serve_many_projections():
    """The decode-step usage: one plan, one workspace, several projections."""
    ml = needs_gpu()
    cfg = WL.TINY
    idx = WL.row_adapters(cfg, "verify")
    ranks = WL.adapter_ranks(cfg)
    ws = ml.Workspace(ml.linear_workspace_bytes(16, 1024, 1024, 4))
    seg_p, _ = ml.plan_segments(dev(idx), dev(ranks), 4, 8, ws)
    for seed in range(3):
        x, W, A, B, rk, _ = _random_case(seed, 16, 512 + 256 * seed, 512, 4, tuple(ranks), r_max=8, nan_pad=False)
        y_ref, _ = _oracle(x, W, A, B, rk, idx, 2.0, OL.VERIFY)
        y = ml.linear(dev_bf16(x), dev_bf16(W), dev_bf16(A), dev_bf16(B), dev(rk), dev(idx), 2.0, ml.VERIFY,
                      ws=ws, seg_offsets_ptr=seg_p)
        assert _rel_err(host_bf16_to_f64(y), y_ref) <= TOL
    assert ws.status() == 0


FULL = [
    (WL.LLAMA8B_R16, None, range(7)),
    (WL.LLAMA8B_HET, None, (1, 4, 6)),
    (WL.QWEN32B_R16, 1, (2, 6)),
    (WL.QWEN32B_R16, 2, (0,)),
    (WL.QWEN32B_R16, 4, (2, 4)),
]


@pytest.mark.parametrize("cfg,k,projs", FULL, ids=lambda v: getattr(v, "name", str(v)))
def test_full_size_sampled_outputs(cfg, k, projs):
    """Workload sizes as benchmarked; 512 sampled outputs per call vs the oracle one by one."""
    ml = needs_gpu()
    ranks = WL.adapter_ranks(cfg)
    for p in projs:
        _, K, N = cfg.projections[p]
        W, A, B, _ = WL.projection_weights(cfg, p)
        Wd, Ad, Bd = dev_bf16(W), dev_bf16(A), dev_bf16(B)
        for mode, name in ((OL.DRAFT, "draft"), (OL.VERIFY, "verify")):
            x = WL.activations(cfg, p, name, k=k)
            idx = WL.row_adapters(cfg, name, k=k)
            M = x.shape[0]
            ws = ml.Workspace(ml.linear_workspace_bytes(M, N, K, cfg.n_adapters))
            y = ml.linear(dev_bf16(x), Wd, Ad, Bd, dev(ranks), dev(idx), cfg.scale, mode, ws=ws)
            yh = host_bf16_to_f64(y)
            assert ws.status() == 0
            g = np.random.default_rng(p)
            rows, cols = g.integers(0, M, 512), g.integers(0, N, 512)
            f = WL.bf16_to_f64
            e = OL.mlora_linear_entries(rows, cols, f(x), f(W), f(A), f(B), ranks, idx, cfg.scale, mode)
            scale_ref = max(np.max(np.abs(e)), 1e-30)
            assert np.max(np.abs(yh[rows, cols] - e)) <= TOL * scale_ref, (cfg.name, p, name)
            assert np.isfinite(yh).all()


def test_prefetch_weights_flag_gives_identical_bits():
    ml = needs_gpu()
    x, W, A, B, rk, idx = _random_case(9, 128, 1024, 4096, 16, (16,) * 16, r_max=16)
    for mode in (ml.DRAFT, ml.VERIFY):
        y0 = _run(ml, x, W, A, B, rk, idx, 2.0, mode)
        y1 = _run(ml, x, W, A, B, rk, idx, 2.0, mode | ml.PREFETCH_WEIGHTS)
        assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))


def test_back_to_back_projections_on_one_stream():
    """Calls that follow one another on a stream overlap their prologues
    (programmatic dependent launch); each still sees its predecessor's output."""
    ml = needs_gpu()
    g = np.random.default_rng(10)
    M, K = 64, 1024
    Ws = [WL.bf16_bits((g.standard_normal((K, K)) / np.sqrt(K)).astype(np.float32)) for _ in range(4)]
    x = WL.bf16_bits(g.standard_normal((M, K)).astype(np.float32))
    ws = ml.Workspace(ml.linear_workspace_bytes(M, K, K, 1))
    h = dev_bf16(x)
    Wd = [dev_bf16(Wb) for Wb in Ws]
    for Wt in Wd:  # y_{i+1} = W_i y_i, each call reading the previous call's output
        h = ml.linear(h, Wt, None, None, None, None, 1.0, ml.DRAFT | ml.PREFETCH_WEIGHTS, ws=ws)
    ref = WL.bf16_to_f64(x)
    for Wb in Ws:
        ref, _ = OL.mlora_linear(ref, WL.bf16_to_f64(Wb), None, None, None, None, 1.0, OL.DRAFT)
        ref = WL.bf16_to_f64(WL.bf16_bits(ref.astype(np.float32)))  # the next layer reads bf16 activations
    assert _rel_err(host_bf16_to_f64(h), ref) <= 2e-2
