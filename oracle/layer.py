"""Oracle for the batched multi-adapter linear layer (float64, numpy).

Test infrastructure only (see the package docstring).

The layer, per token row m with adapter a = adapter_idx[m] and rank r = rank_of[a]:

    y[m] = W x[m]                                          draft  (LoRA off)
    y[m] = W x[m] + scale * B_a[:, :r] (A_a[:r, :] x[m])   verify (LoRA on)

"Multi-LoRA Serving in Practice", section "Core Principle: Shared Base Model,
Per-Request Adapter Selection" gives output = W·x + scale · B(A·x) with the
request naming its adapter; the InvisibleLoRA abstract gives the two modes
(a LoRA-off draft pass and a LoRA-on verify pass).

Layouts (a reading; the pages fix none): row-major, W [N, K] (out x in),
A_stack [n_adapters, r_max, K], B_stack [n_adapters, N, r_max], x [M, K],
y [M, N].  Only the first rank_of[a] rows of A_a and columns of B_a are read.

Readings where the pages are silent:
  * adapter_idx = -1 means "base model only" for that row.
  * An adapter index outside [-1, n_adapters) or a rank outside [0, r_max] is
    invalid input: the row (or adapter) runs without the low-rank term and a
    status bit is raised.
"""
from __future__ import annotations

import numpy as np

DRAFT = 0
VERIFY = 1

# Status bits, as documented for the library's device status word.
STATUS_BAD_ADAPTER = 1 << 0
STATUS_BAD_RANK = 1 << 1


def effective_ranks(rank_of, r_max: int):
    """Ranks with invalid entries (outside [0, r_max]) replaced by 0, plus status."""
    r = np.asarray(rank_of, dtype=np.int64)
    bad = (r < 0) | (r > r_max)
    return np.where(bad, 0, r), (STATUS_BAD_RANK if bad.any() else 0)


def row_buckets(adapter_idx, n_adapters: int):
    """Bucket of each row: its adapter, or n_adapters ("no adapter") for -1 and
    for invalid indices.  Returns (bucket, status)."""
    idx = np.asarray(adapter_idx, dtype=np.int64)
    bad = (idx < -1) | (idx >= n_adapters)
    bucket = np.where((idx < 0) | bad, n_adapters, idx)
    return bucket, (STATUS_BAD_ADAPTER if bad.any() else 0)


def plan_segments(adapter_idx, n_adapters: int):
    """Group rows by adapter: a stable counting sort.

    The InvisibleLoRA abstract notes that requests are partitioned across the
    active adapters; "Multi-LoRA Serving in Practice", section "4. Batching",
    calls for aggregating requests of the same adapter.  Rows of bucket b
    (adapter b, or n_adapters for rows without an adapter) occupy sorted
    positions seg_offsets[b] .. seg_offsets[b+1]-1, in increasing row order.

    Returns (seg_offsets int32 [n_adapters + 2], perm int32 [M] with
    perm[sorted position] = row, status).
    """
    bucket, status = row_buckets(adapter_idx, n_adapters)
    M = bucket.shape[0]
    seg_offsets = np.zeros(n_adapters + 2, dtype=np.int32)
    perm = []
    for b in range(n_adapters + 1):
        rows = [m for m in range(M) if bucket[m] == b]
        perm.extend(rows)
        seg_offsets[b + 1] = seg_offsets[b] + len(rows)
    return seg_offsets, np.asarray(perm, dtype=np.int32), status


def shrink(x, A_stack, rank_of, adapter_idx):
    """Low-rank activations T[m, j] = sum_k A_a[j, k] x[m, k] for j < rank_of[a].

    Entries j >= rank_of[a], and every entry of rows without a (valid)
    adapter, are 0.  Returns (T float64 [M, r_max], status).
    """
    x = np.asarray(x, dtype=np.float64)
    A = np.asarray(A_stack, dtype=np.float64)
    n_ad, r_max, _ = A.shape
    ranks, st_r = effective_ranks(rank_of, r_max)
    bucket, st_a = row_buckets(adapter_idx, n_ad)
    T = np.zeros((x.shape[0], r_max), dtype=np.float64)
    for a in range(n_ad):
        rows = np.nonzero(bucket == a)[0]
        r = int(ranks[a])
        if rows.size == 0 or r == 0:
            continue
        T[rows, :r] = x[rows] @ A[a, :r, :].T
    return T, st_r | st_a


def mlora_linear(x, W, A_stack, B_stack, rank_of, adapter_idx, scale: float, mode: int):
    """Layer output y float64 [M, N] (not rounded) and status.

    Rows are grouped by adapter and each group goes through one BLAS product;
    grouping changes nothing but the speed of this oracle.
    """
    x = np.asarray(x, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    y = x @ W.T
    if mode == DRAFT:
        return y, 0
    if A_stack is None or B_stack is None:
        return y, 0
    A = np.asarray(A_stack, dtype=np.float64)
    B = np.asarray(B_stack, dtype=np.float64)
    n_ad, r_max, _ = A.shape
    ranks, st_r = effective_ranks(rank_of, r_max)
    bucket, st_a = row_buckets(adapter_idx, n_ad)
    for a in range(n_ad):
        rows = np.nonzero(bucket == a)[0]
        r = int(ranks[a])
        if rows.size == 0 or r == 0:
            continue
        t = x[rows] @ A[a, :r, :].T            # [rows, r]
        y[rows] += float(scale) * (t @ B[a, :, :r].T)
    return y, st_r | st_a


def mlora_linear_entries(rows, cols, x, W, A_stack, B_stack, rank_of, adapter_idx, scale: float, mode: int):
    """Selected outputs y[rows[i], cols[i]] one by one, for spot checks at
    sizes where the full product is too slow on a CPU."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    out = np.empty(rows.shape[0], dtype=np.float64)
    n_ad = None if A_stack is None else A_stack.shape[0]
    r_max = None if A_stack is None else A_stack.shape[1]
    ranks = None if A_stack is None else effective_ranks(rank_of, r_max)[0]
    bucket = None if A_stack is None else row_buckets(adapter_idx, n_ad)[0]
    for i, (m, n) in enumerate(zip(rows, cols)):
        xm = np.asarray(x[m], dtype=np.float64)
        v = float(np.dot(np.asarray(W[n], dtype=np.float64), xm))
        if mode == VERIFY and A_stack is not None:
            a = int(bucket[m])
            if a < n_ad and ranks[a] > 0:
                r = int(ranks[a])
                t = np.asarray(A_stack[a, :r, :], dtype=np.float64) @ xm
                v += float(scale) * float(np.dot(np.asarray(B_stack[a, n, :r], dtype=np.float64), t))
        out[i] = v
    return out
