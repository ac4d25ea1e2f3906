"""Oracle: the contiguous in-seq-split comparator.

Test infrastructure only (see the package docstring).

Source: "[DeepSeek v3.2] 上下文并行详解", section 4 part 1: the older context-parallel mode cuts
each prompt into contiguous chunks, one per rank (8000 tokens on 8 ranks: rank 0 gets tokens
0-999, rank 1 gets 1000-1999, ...); with two requests A (8000) and B (800), rank 0 gets A's
0-999 and B's 0-99; with a coarse chunk a 5-token request keeps only rank 0 busy.

Reading: chunk = max(ceil(L/sp), granularity) tokens per rank and request; granularity 1 gives
the page's per-request chunks, a larger granularity gives its coarse-chunk remark.
"""
from __future__ import annotations

import numpy as np


def in_seq_positions(length: int, sp: int, rank: int, granularity: int = 1) -> np.ndarray:
    chunk = max(-(-int(length) // sp), int(granularity))
    lo = min(rank * chunk, length)
    hi = min((rank + 1) * chunk, length)
    return np.arange(lo, hi, dtype=np.int64)


def in_seq_split(lengths, sp: int, rank: int, granularity: int = 1):
    """(bid, pos) of every token rank `rank` holds under in-seq-split, request by request."""
    bid, pos = [], []
    for b, L in enumerate(lengths):
        p = in_seq_positions(L, sp, rank, granularity)
        bid.append(np.full(len(p), b, dtype=np.int64))
        pos.append(p)
    if not bid:
        return np.zeros(0, np.int64), np.zeros(0, np.int64)
    return np.concatenate(bid), np.concatenate(pos)


def causal_pairs(pos: np.ndarray) -> int:
    """Causal (query, key) pairs a set of queries scans: sum of (pos + 1)."""
    return int(np.sum(np.asarray(pos, dtype=np.int64) + 1))
