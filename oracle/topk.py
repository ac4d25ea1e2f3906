"""Oracle: per-query top-k of a score row, lowest index wins ties.

Test infrastructure only (see the package docstring).

"[RFC]: Parallel strategy for Deepseek v3.2 like models" says only that the indexer selects the
history top-K keys of each query. The rule used: the k indices s in [0, L) with the largest
score; equal scores go to the lower index; -0.0 equals +0.0; when L <= k every index is taken.
The result is listed in ascending index order and padded with -1 up to k entries (the set is the
contract; the order makes arrays comparable).

Method: one full stable sort of the pairs (-score, index), then the first k, then ascending.
The comparison happens in the precision of the array given (fp64 oracle scores, or fp32 when a
caller rounds them first).
"""
from __future__ import annotations

import numpy as np


def topk_indices(scores, k: int) -> np.ndarray:
    scores = np.asarray(scores)
    # canonical zero: -0.0 and +0.0 must compare equal and fall to the index tie-break
    scores = np.where(scores == 0, np.zeros((), dtype=scores.dtype), scores)
    idx = np.arange(scores.shape[0])
    order = np.lexsort((idx, -scores))      # primary: larger score first; then lower index
    chosen = np.sort(order[:k])
    out = np.full(k, -1, dtype=np.int64)
    out[:chosen.shape[0]] = chosen
    return out


def topk_rows(score_rows, k: int) -> np.ndarray:
    return np.stack([topk_indices(r, k) for r in score_rows]) if score_rows else \
        np.zeros((0, k), dtype=np.int64)
