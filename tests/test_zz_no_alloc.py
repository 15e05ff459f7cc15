"""The allocation-free layer entry point (mlora_linear_noalloc).

Some callers cannot allocate device memory (a plugin whose host framework
owns every device buffer, or code with a memory budget fixed at start-up), so
they cannot give mlora_linear a workspace.  mlora_linear_noalloc keeps its
scratch in an array compiled into the library.  These tests call it through
the C ABI twice in a row, with different inputs, and check each output
against mlora_linear's within the layer tolerance used by every GPU test.
This file is collected last so that a run stopping at the first failure has
run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from tests.gpu_util import dev, dev_bf16, needs_gpu

pytestmark = pytest.mark.gpu
TOL = 1e-2


def _case(seed, M, N, K, n_ad, r):
    g = np.random.default_rng(seed)
    import workloads as WL
    x = WL.bf16_bits(g.standard_normal((M, K)).astype(np.float32))
    W = WL.bf16_bits((g.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32))
    A = WL.bf16_bits((g.standard_normal((n_ad, r, K)) / np.sqrt(K)).astype(np.float32))
    B = WL.bf16_bits((g.standard_normal((n_ad, N, r)) / np.sqrt(r)).astype(np.float32))
    idx = g.integers(-1, n_ad, M).astype(np.int32)
    ranks = np.full(n_ad, r, np.int32)
    return dev_bf16(x), dev_bf16(W), dev_bf16(A), dev_bf16(B), dev(ranks), dev(idx)


def _rel(a, b):
    a = a.float().cpu().numpy().astype(np.float64)
    b = b.float().cpu().numpy().astype(np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-30))


def _oracle(case, mode):
    import workloads as WL
    from oracle import layer as OL
    x, W, A, B, rk, idx = case
    f = lambda t: t.float().cpu().numpy().astype(np.float64)  # noqa: E731  (bf16 values, exact in float64)
    y, _ = OL.mlora_linear(f(x), f(W), f(A), f(B), rk.cpu().numpy(), idx.cpu().numpy(), 2.0, mode)
    return y


def _rel_np(a, b):
    a = a.float().cpu().numpy().astype(np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-30))


@pytest.mark.parametrize("mode_name", ["draft", "verify"])
def test_noalloc_matches_workspace_entry_point_on_two_calls(mode_name):
    ml = needs_gpu()
    mode = ml.DRAFT if mode_name == "draft" else ml.VERIFY
    # the second case has more than 512 rows: the GEMM takes two token groups
    cases = [_case(1, 128, 1024, 4096, 16, 16), _case(2, 700, 1024, 1024, 8, 16)]
    refs = []
    for x, W, A, B, rk, idx in cases:
        refs.append(ml.linear(x, W, A, B, rk, idx, 2.0, mode))
    outs = [ml.linear_noalloc(x, W, A, B, rk, idx, 2.0, mode) for (x, W, A, B, rk, idx) in cases]
    torch.cuda.synchronize()
    for case, y, y_ref in zip(cases, outs, refs):
        assert _rel(y, y_ref) <= TOL
        assert _rel_np(y, _oracle(case, mode)) <= TOL


def test_noalloc_refuses_sizes_beyond_its_array():
    ml = needs_gpu()
    lib = ml.library()
    x, W, A, B, rk, idx = _case(3, 8, 128, 64, 4, 8)
    big = ml.NOALLOC_MAX_ROWS + 1
    st = lib.mlora_linear_noalloc(x.data_ptr(), big, 64, W.data_ptr(), 128, A.data_ptr(), B.data_ptr(), 4, 8,
                                  rk.data_ptr(), idx.data_ptr(), ctypes.c_float(2.0), ml.VERIFY, x.data_ptr(), None)
    assert st == 2  # MLORA_ERR_SHAPE
