"""Pins for the hybrid KV cache oracle (oracle.kvcache).

The oracle places each pass's K/V rows in a paged cache.  Its pins: cases
worked by hand (tests/golden/kv_hand_example.json), the identity with a dense
[B, positions, H, D] cache when every request owns consecutive blocks, the
read-back through the block table, that nothing else in the cache changes,
and one whole decode cycle of the hybrid cache (drafts write speculative
entries, the verify pass overwrites every one of them, the commit keeps the
accepted prefix).
"""
import json
import os

import numpy as np

from oracle import kvcache as OK

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_hand_example.json")


def _run_case(c):
    nb, bs, H, D = c["num_blocks"], c["block_size"], c["H"], c["D"]
    kc = np.full((nb, bs, H, D), 65535, np.uint16)
    vc = kc.copy()
    bt = np.array(c["block_table"], np.int32)
    y = np.array(c["y"], np.uint16)
    return OK.kv_write(y, c["k_col"], c["v_col"], H, D, bt, np.array(c["seq_len"], np.int32), c["rows_per_req"],
                       c["t0"], kc, vc), kc, vc


def test_hand_worked_cases():
    g = json.load(open(GOLDEN))
    for c in g["cases"]:
        (k2, v2, st), k0, v0 = _run_case(c)
        assert st == c["status"], c["why"]
        ek, ev = k0.copy(), v0.copy()
        for w in c["writes"]:
            ek[w["block"], w["offset"]] = np.array(w["k"], np.uint16)
            ev[w["block"], w["offset"]] = np.array(w["v"], np.uint16)
        assert np.array_equal(k2, ek) and np.array_equal(v2, ev), c["why"]
    cm = g["commit"]
    assert OK.commit(np.array(cm["seq_len"]), np.array(cm["accepted"])).tolist() == cm["expected"]


def _random_setup(g, B, H, D, bs, max_blocks, extra_blocks=3):
    nb = B * max_blocks + extra_blocks
    perm = g.permutation(nb)[: B * max_blocks].reshape(B, max_blocks).astype(np.int32)
    kc = g.integers(0, 65536, (nb, bs, H, D), dtype=np.uint16)
    vc = g.integers(0, 65536, (nb, bs, H, D), dtype=np.uint16)
    return perm, kc, vc


def test_dense_equivalence_with_consecutive_blocks():
    """Request b owning blocks [b n, (b + 1) n) makes the paged cache a dense
    [B, n * block_size, H, D] array indexed by (request, position)."""
    g = np.random.default_rng(1)
    B, H, D, bs, n = 5, 2, 4, 4, 3
    bt = np.arange(B * n, dtype=np.int32).reshape(B, n)
    kc = g.integers(0, 65536, (B * n, bs, H, D), dtype=np.uint16)
    vc = g.integers(0, 65536, (B * n, bs, H, D), dtype=np.uint16)
    seq = g.integers(0, n * bs - 3, B).astype(np.int32)
    k = 2
    ld, kcol, vcol = 3 * H * D, H * D, 2 * H * D
    y = g.integers(0, 65536, (B * (k + 1), ld), dtype=np.uint16)
    k2, v2, st = OK.kv_write(y, kcol, vcol, H, D, bt, seq, k + 1, 0, kc, vc)
    assert st == 0
    dk, dv = kc.reshape(B, n * bs, H, D).copy(), vc.reshape(B, n * bs, H, D).copy()
    for m in range(B * (k + 1)):
        b, t = divmod(m, k + 1)
        dk[b, seq[b] + t] = y[m, kcol:kcol + H * D].reshape(H, D)
        dv[b, seq[b] + t] = y[m, vcol:vcol + H * D].reshape(H, D)
    assert np.array_equal(k2.reshape(B, n * bs, H, D), dk) and np.array_equal(v2.reshape(B, n * bs, H, D), dv)


def test_read_back_and_nothing_else_changes():
    g = np.random.default_rng(2)
    B, H, D, bs, mb = 7, 3, 2, 2, 5
    bt, kc, vc = _random_setup(g, B, H, D, bs, mb)
    seq = g.integers(0, mb * bs - 4, B).astype(np.int32)
    k = 3
    ld = 40
    kcol, vcol = 5, 5 + H * D  # any column offsets
    y = g.integers(0, 65536, (B * (k + 1), ld), dtype=np.uint16)
    k2, v2, st = OK.kv_write(y, kcol, vcol, H, D, bt, seq, k + 1, 0, kc, vc)
    assert st == 0
    for b in range(B):
        pos = [int(seq[b]) + t for t in range(k + 1)]
        rk, rv = OK.read_back(k2, v2, bt, b, pos, bs)
        rows = y[b * (k + 1):(b + 1) * (k + 1)]
        assert np.array_equal(rk, rows[:, kcol:kcol + H * D].reshape(k + 1, H, D))
        assert np.array_equal(rv, rows[:, vcol:vcol + H * D].reshape(k + 1, H, D))
    changed = np.any((k2 != kc).reshape(k2.shape[0], bs, -1), axis=2)
    assert changed.sum() <= B * (k + 1)  # (a written row may equal the old one by chance)
    touched = {(int(bt[b, (seq[b] + t) // bs]), int((seq[b] + t) % bs)) for b in range(B) for t in range(k + 1)}
    for blk, off in zip(*np.nonzero(changed)):
        assert (int(blk), int(off)) in touched


def test_one_hybrid_decode_cycle():
    """k draft steps write speculative entries at L..L+k-1; the verify pass
    overwrites L..L+k; the commit after n kept drafts makes L+n+1 committed,
    and each committed entry holds the verify pass's (LoRA-on) row."""
    g = np.random.default_rng(3)
    B, H, D, bs, mb, k = 4, 2, 2, 4, 4, 3
    bt, kc, vc = _random_setup(g, B, H, D, bs, mb)
    L = g.integers(0, mb * bs - k - 2, B).astype(np.int32)
    ld, kcol, vcol = 2 * H * D, 0, H * D
    drafts = []
    for t in range(k):  # the LoRA-off steps
        yd = g.integers(0, 65536, (B, ld), dtype=np.uint16)
        drafts.append(yd)
        kc, vc, st = OK.kv_write(yd, kcol, vcol, H, D, bt, L, 1, t, kc, vc)
        assert st == 0
    for b in range(B):  # the drafter reads its own speculative entries
        rk, _ = OK.read_back(kc, vc, bt, b, [int(L[b]) + t for t in range(k)], bs)
        assert np.array_equal(rk, np.stack([drafts[t][b, :H * D].reshape(H, D) for t in range(k)]))
    yv = g.integers(0, 65536, (B * (k + 1), ld), dtype=np.uint16)  # the LoRA-on pass
    kc, vc, st = OK.kv_write(yv, kcol, vcol, H, D, bt, L, k + 1, 0, kc, vc)
    assert st == 0
    n = g.integers(0, k + 1, B)
    L2 = OK.commit(L, n)
    assert np.array_equal(L2, L + n + 1)
    for b in range(B):
        pos = list(range(int(L[b]), int(L2[b])))
        rk, rv = OK.read_back(kc, vc, bt, b, pos, bs)
        rows = yv[b * (k + 1):b * (k + 1) + len(pos)]
        assert np.array_equal(rk, rows[:, :H * D].reshape(-1, H, D))
        assert np.array_equal(rv, rows[:, H * D:].reshape(-1, H, D))
        # no speculative (LoRA-off) entry survives anywhere in L..L+k
        rk_all, _ = OK.read_back(kc, vc, bt, b, [int(L[b]) + t for t in range(k + 1)], bs)
        assert np.array_equal(rk_all, yv[b * (k + 1):(b + 1) * (k + 1), :H * D].reshape(-1, H, D))


def test_rows_past_the_batch_and_empty_pass():
    g = np.random.default_rng(4)
    bt, kc, vc = _random_setup(g, 2, 1, 2, 2, 2)
    seq = np.array([0, 1], np.int32)
    y = np.zeros((0, 4), np.uint16)
    k2, v2, st = OK.kv_write(y, 0, 2, 1, 2, bt, seq, 1, 0, kc, vc)
    assert st == 0 and np.array_equal(k2, kc) and np.array_equal(v2, vc)
