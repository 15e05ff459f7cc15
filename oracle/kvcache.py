"""Oracle for the hybrid KV cache: where each pass's K and V rows go in the
paged cache of the LoRA-on target model (numpy, integer indexing and 16-bit
word copies only).

Test infrastructure only (see the package docstring).

The InvisibleLoRA abstract describes one KV cache for both models: the
LoRA-off drafter writes its speculative K/V entries into the target's cache,
the LoRA-on verification pass overwrites those entries, and the drafter
therefore reads LoRA-conditioned K/V for the committed prefix.  The pages give
no layout; the readings taken:

  * A paged cache: K and V each [num_blocks, block_size, H, D] of bf16 words;
    request b's position `pos` lives in block block_table[b, pos // block_size]
    at offset pos % block_size.  A block id outside [0, num_blocks), or a
    position past the request's table, is an invalid slot: the row is not
    written and status bit 7 is raised.
  * seq_len[b] counts request b's committed tokens, whose K/V are in the cache
    with LoRA-on values; a negative seq_len marks an unused request slot,
    whose rows are skipped without a status.
  * One decode cycle of draft length k: the token pending at position L =
    seq_len[b] and k - 1 drafts run through the LoRA-off pass one step at a
    time (draft step t writes position L + t), then the pending token and all
    k drafts run through the LoRA-on pass as k + 1 rows per request
    (row b (k + 1) + t writes position L + t, overwriting the drafter's
    entries).  After the accept step keeps n drafts, the committed length is
    L + n + 1; the slots past it hold entries that the next cycle overwrites.
  * The K and V rows come from the fused q|k|v projection's output y: K of
    row m is y[m, k_col : k_col + H D], V is y[m, v_col : v_col + H D], each
    read as H heads of D contiguous values.

Every function returns new arrays; the inputs are not modified.
"""
from __future__ import annotations

import numpy as np

BAD_SLOT = 1 << 7  # status bit: a row whose slot is outside the cache or its table


def slot_of(block_table, seq_len, b: int, t: int, block_size: int, num_blocks: int):
    """(block, offset) of request b's position seq_len[b] + t, or None when
    the position or its block is outside the cache."""
    pos = int(seq_len[b]) + int(t)
    j = pos // block_size
    if pos < 0 or j >= block_table.shape[1]:
        return None
    blk = int(block_table[b, j])
    if blk < 0 or blk >= num_blocks:
        return None
    return blk, pos % block_size


def kv_write(y, k_col: int, v_col: int, H: int, D: int, block_table, seq_len, rows_per_req: int, t0: int,
             k_cache, v_cache):
    """Write the K and V rows of one pass into the paged cache.

    y            uint16 [M, ld]: the fused projection's output, bf16 words;
    rows_per_req 1 for a draft step, k + 1 for the verify pass: row m belongs
                 to request m // rows_per_req at step t = m % rows_per_req;
    t0           the draft step (draft pass) or 0 (verify pass): row m writes
                 position seq_len[b] + t0 + t.
    Returns (k_cache', v_cache', status)."""
    y = np.asarray(y, dtype=np.uint16)
    kc = np.array(k_cache, dtype=np.uint16, copy=True)
    vc = np.array(v_cache, dtype=np.uint16, copy=True)
    num_blocks, block_size = kc.shape[0], kc.shape[1]
    status = 0
    M = y.shape[0]
    for m in range(M):
        b, t = divmod(m, rows_per_req)
        if b >= len(seq_len) or int(seq_len[b]) < 0:
            continue  # unused request slot (or a row past the batch)
        where = slot_of(block_table, seq_len, b, t0 + t, block_size, num_blocks)
        if where is None:
            status |= BAD_SLOT
            continue
        blk, off = where
        kc[blk, off] = y[m, k_col:k_col + H * D].reshape(H, D)
        vc[blk, off] = y[m, v_col:v_col + H * D].reshape(H, D)
    return kc, vc, status


def commit(seq_len, accepted):
    """Committed lengths after the accept step: L + n + 1 for each used
    request slot (the pending token and the n kept drafts), unchanged for an
    unused one."""
    s = np.array(seq_len, dtype=np.int64, copy=True)
    for b in range(len(s)):
        if s[b] >= 0:
            s[b] += int(accepted[b]) + 1
    return s.astype(np.int32)


def read_back(k_cache, v_cache, block_table, b: int, positions, block_size: int):
    """K and V of request b at the given positions, through its block table
    ([len(positions), H, D] each): what the attention of either model reads."""
    ks, vs = [], []
    for pos in positions:
        blk = int(block_table[b, pos // block_size])
        ks.append(np.asarray(k_cache)[blk, pos % block_size])
        vs.append(np.asarray(v_cache)[blk, pos % block_size])
    return np.array(ks), np.array(vs)
