"""GPU parity of the hybrid KV cache (mlora_kv_write, mlora_kv_commit) with
the oracle (oracle.kvcache).  The copy moves 16-bit words, so the caches must
match the oracle's bit for bit, including every slot the pass must leave
alone, and the status bits must match."""
import numpy as np
import pytest
import torch

from oracle import kvcache as OK
from tests.gpu_util import dev, needs_gpu

pytestmark = pytest.mark.gpu


def _u16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _bf16(a):
    return dev(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def _setup(g, B, H, D, bs, max_blocks, extra=5, unalloc=0.0):
    nb = B * max_blocks + extra
    bt = g.permutation(nb)[: B * max_blocks].reshape(B, max_blocks).astype(np.int32)
    if unalloc:
        bt[g.random(bt.shape) < unalloc] = -1
    kc = g.integers(0, 65536, (nb, bs, H, D), dtype=np.uint16)
    vc = g.integers(0, 65536, (nb, bs, H, D), dtype=np.uint16)
    return bt, kc, vc


def _check(ml, y, k_col, v_col, H, D, bt, seq, rpr, t0, kc, vc, y_dev=None):
    ek, ev, est = OK.kv_write(y, k_col, v_col, H, D, bt, seq, rpr, t0, kc, vc)
    ws = ml.Workspace(ml.kv_workspace_bytes())
    kd, vd = _bf16(kc), _bf16(vc)
    ml.kv_write(_bf16(y) if y_dev is None else y_dev, k_col, v_col, H, D, dev(bt), dev(seq), rpr, t0, kd, vd, ws=ws)
    assert ws.status() == est
    assert np.array_equal(_u16(kd), ek) and np.array_equal(_u16(vd), ev)
    return ek, ev


@pytest.mark.parametrize("k", [1, 2, 4])
def test_verify_pass_32b_shapes(k):
    """The 32B block's fused q|k|v output (q 5120, k 1024, v 1024 columns; 8
    KV heads of 128) for 128 requests at k + 1 rows each, 16-token blocks."""
    ml = needs_gpu()
    g = np.random.default_rng(k)
    B, H, D, bs, mb = 128, 8, 128, 16, 8
    bt, kc, vc = _setup(g, B, H, D, bs, mb)
    seq = g.integers(0, mb * bs - k - 1, B).astype(np.int32)
    y = g.integers(0, 65536, (B * (k + 1), 5120 + 2048), dtype=np.uint16)
    _check(ml, y, 5120, 6144, H, D, bt, seq, k + 1, 0, kc, vc)


def test_one_decode_cycle_on_the_gpu():
    """Draft steps, the verify pass and the commit, chained on the device as in
    a decode cycle, against the oracle's cycle."""
    ml = needs_gpu()
    g = np.random.default_rng(7)
    B, H, D, bs, mb, k = 64, 8, 128, 16, 6, 4
    bt, kc, vc = _setup(g, B, H, D, bs, mb)
    L = g.integers(0, mb * bs - 2 * k - 2, B).astype(np.int32)
    L[3] = -1  # an unused request slot
    ld = 3 * H * D
    ws = ml.Workspace(ml.kv_workspace_bytes())
    kd, vd, bt_d, seq_d = _bf16(kc), _bf16(vc), dev(bt), dev(L)
    ek, ev = kc, vc
    for t in range(k):
        yd = g.integers(0, 65536, (B, ld), dtype=np.uint16)
        ml.kv_write(_bf16(yd), H * D, 2 * H * D, H, D, bt_d, seq_d, 1, t, kd, vd, ws=ws)
        ek, ev, _ = OK.kv_write(yd, H * D, 2 * H * D, H, D, bt, L, 1, t, ek, ev)
    yv = g.integers(0, 65536, (B * (k + 1), ld), dtype=np.uint16)
    ml.kv_write(_bf16(yv), H * D, 2 * H * D, H, D, bt_d, seq_d, k + 1, 0, kd, vd, ws=ws)
    ek, ev, _ = OK.kv_write(yv, H * D, 2 * H * D, H, D, bt, L, k + 1, 0, ek, ev)
    acc = g.integers(0, k + 1, B).astype(np.int32)
    ml.kv_commit(dev(acc), seq_d)
    L2 = OK.commit(L, acc)
    # the next cycle's first draft step lands after the committed prefix
    yn = g.integers(0, 65536, (B, ld), dtype=np.uint16)
    ml.kv_write(_bf16(yn), H * D, 2 * H * D, H, D, bt_d, seq_d, 1, 0, kd, vd, ws=ws)
    ek, ev, _ = OK.kv_write(yn, H * D, 2 * H * D, H, D, bt, L2, 1, 0, ek, ev)
    assert ws.status() == 0
    assert np.array_equal(seq_d.cpu().numpy(), L2)
    assert np.array_equal(_u16(kd), ek) and np.array_equal(_u16(vd), ev)


def test_invalid_slots_and_unused_requests():
    ml = needs_gpu()
    g = np.random.default_rng(11)
    B, H, D, bs, mb, k = 16, 2, 64, 4, 3, 2
    bt, kc, vc = _setup(g, B, H, D, bs, mb, unalloc=0.2)
    bt[0, 0] = bt.max() + 10  # a block id past the cache
    seq = g.integers(0, mb * bs, B).astype(np.int32)  # some positions run past the table
    seq[5] = -1
    y = g.integers(0, 65536, (B * (k + 1), 3 * H * D), dtype=np.uint16)
    seq[0] = 0
    _check(ml, y, H * D, 2 * H * D, H, D, bt, seq, k + 1, 0, kc, vc)


@pytest.mark.parametrize("H,D,k_col,v_col,ld", [(1, 3, 1, 7, 11), (3, 5, 0, 15, 40), (2, 8, 3, 21, 40)])
def test_unaligned_rows_take_the_word_copy(H, D, k_col, v_col, ld):
    """Row segments that do not start on 16 bytes (odd columns, odd H*D)."""
    ml = needs_gpu()
    g = np.random.default_rng(H * 100 + D)
    B, bs, mb, k = 9, 3, 4, 3
    bt, kc, vc = _setup(g, B, H, D, bs, mb)
    seq = g.integers(0, mb * bs - k - 1, B).astype(np.int32)
    y = g.integers(0, 65536, (B * (k + 1), ld), dtype=np.uint16)
    _check(ml, y, k_col, v_col, H, D, bt, seq, k + 1, 0, kc, vc)


def test_partial_batch_and_empty_pass():
    """M below B * rows_per_req (the last request's rows cut short) and M = 0."""
    ml = needs_gpu()
    g = np.random.default_rng(5)
    B, H, D, bs, mb, k = 6, 4, 32, 8, 2, 3
    bt, kc, vc = _setup(g, B, H, D, bs, mb)
    seq = g.integers(0, mb * bs - k - 1, B).astype(np.int32)
    y = g.integers(0, 65536, (B * (k + 1) - 2, 2 * H * D), dtype=np.uint16)
    _check(ml, y, 0, H * D, H, D, bt, seq, k + 1, 0, kc, vc)
    _check(ml, np.zeros((0, 2 * H * D), np.uint16), 0, H * D, H, D, bt, seq, 1, 0, kc, vc)


def test_output_of_the_layer_feeds_the_cache():
    """mlora_linear_sliced's q|k|v output written straight into the cache: the
    cache holds exactly the K/V columns of the layer output."""
    ml = needs_gpu()
    import workloads as WL
    g = np.random.default_rng(9)
    M, K = 64, 512
    Nq, Nkv, H, D = 256, 128, 2, 64
    W = WL._normal_bf16(g, (Nq + 2 * Nkv, K), 1.0 / np.sqrt(K))
    x = WL._normal_bf16(g, (M, K), 1.0)
    y = ml.linear(_bf16(x), _bf16(W), None, None, None, None, 1.0, ml.DRAFT)
    bt, kc, vc = _setup(g, M, H, D, 16, 2)
    seq = g.integers(0, 31, M).astype(np.int32)
    _check(ml, _u16(y), Nq, Nq + Nkv, H, D, bt, seq, 1, 0, kc, vc, y_dev=y)
