"""Oracle: all-gathered KV buffer -> logical token order (the rerange).

Test infrastructure only (see the package docstring).

Source: "[DeepSeek v3.2] 上下文并行详解", section 2.C (cp_all_gather_rerange_output) and
section 4 part 3 step B: after the all-gather, rows sit rank by rank ("T0,T4, T1,T5, ..."), and
the rerange puts them back in the logical order T0, T1, T2, ... because the top-k selection needs
the KV logically contiguous.

Reading taken where the page is silent: the page gives the rank-major order but not whether
each rank's block is padded. Both layouts are modelled: padded (every rank's block starts at
rank * stride, stride >= ceil(N/sp), the equal-size all-gather) and packed (blocks back to back,
stride = 0).
"""
from __future__ import annotations

import numpy as np

from .split import shard_tokens


def rank_offsets(n_tokens: int, sp: int, stride: int = 0) -> np.ndarray:
    """Row where each rank's block starts in the gathered buffer."""
    if stride > 0:
        return np.arange(sp, dtype=np.int64) * stride
    sizes = [len(shard_tokens(n_tokens, sp, q)) for q in range(sp)]
    return np.concatenate([[0], np.cumsum(sizes)[:-1]]).astype(np.int64)


def all_gather(shards, stride: int = 0) -> np.ndarray:
    """Concatenate the ranks' local rows rank by rank; with stride > 0 pad each block with zeros."""
    if stride <= 0:
        return np.concatenate(shards, axis=0)
    blocks = []
    for s in shards:
        pad = np.zeros((stride - s.shape[0],) + s.shape[1:], dtype=s.dtype)
        blocks.append(np.concatenate([s, pad], axis=0))
    return np.concatenate(blocks, axis=0)


def rerange(gathered: np.ndarray, n_tokens: int, sp: int, stride: int = 0) -> np.ndarray:
    """Undo the rank-major layout: rank q's j-th local row is token q + j*sp."""
    off = rank_offsets(n_tokens, sp, stride)
    out = np.empty((n_tokens,) + gathered.shape[1:], dtype=gathered.dtype)
    for q in range(sp):
        tokens = shard_tokens(n_tokens, sp, q)
        out[tokens] = gathered[off[q]:off[q] + len(tokens)]
    return out


def rerange_into_pages(gathered: np.ndarray, cu, sp: int, stride: int, block_table,
                       page_size: int, pool: np.ndarray) -> np.ndarray:
    """The rerange fused with the write of the KV cache: logical token g of request b (position
    s = g - cu[b]) goes straight to pool row block_table[b, s // page_size] * page_size +
    s % page_size instead of row g of a contiguous buffer. Rows of the pool that no token maps to
    keep their contents. ("[RFC]: Parallel strategy for Deepseek v3.2 like models", "New
    proposal": the KV is all-gathered before the KV-cache update step; "[DeepSeek v3.2]
    上下文并行详解", section 4 part 3 step B for the rerange.)"""
    cu = np.asarray(cu, dtype=np.int64)
    table = np.asarray(block_table, dtype=np.int64)
    logical = rerange(gathered, int(cu[-1]), sp, stride)
    out = pool.copy()
    for b in range(len(cu) - 1):
        for s in range(int(cu[b + 1] - cu[b])):
            page = table[b, s // page_size]
            out[page * page_size + s % page_size] = logical[cu[b] + s]
    return out


def cache_local_into_pages(local_rows: np.ndarray, cu, sp: int, rank: int, block_table,
                           page_size: int, pool: np.ndarray) -> np.ndarray:
    """After attention a rank drops the global KV and its cache keeps only the tokens it owns
    ("[DeepSeek v3.2] 上下文并行详解", section 4 part 3 step D: with CP = 4, rank 1 stores only
    K1 and K5 in its cache pool for the decode steps). local_rows[t] is the rank's t-th token,
    flattened index g = rank + t*sp. Reading taken where the page is silent: the rank's cache of
    request b lists that request's tokens on this rank in order, the j-th of them in slot j, and
    slot j lives in row block_table[b, j // page_size] * page_size + j % page_size of the rank's
    pool. Rows of the pool that no token maps to keep their contents."""
    cu = np.asarray(cu, dtype=np.int64)
    table = np.asarray(block_table, dtype=np.int64)
    tokens = shard_tokens(int(cu[-1]), sp, rank)
    out = pool.copy()
    for b in range(len(cu) - 1):
        mine = [t for t, g in enumerate(tokens) if cu[b] <= g < cu[b + 1]]
        for j, t in enumerate(mine):
            page = table[b, j // page_size]
            out[page * page_size + j % page_size] = local_rows[t]
    return out
