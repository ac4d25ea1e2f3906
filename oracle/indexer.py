"""Oracle: lightning-indexer scores over the causal history.

Test infrastructure only (see the package docstring).

Definition (DeepSeek-V3.2 DSA lightning indexer; "[RFC]: Parallel strategy for Deepseek v3.2
like models" names this scan the model's bottleneck and explains that each query loops over its
whole history to pick the top-K keys):

    I[t, s] = sum_h  w[t, h] * ReLU( sum_d q_idx[t, h, d] * k_idx[row(b_t, s), d] ),
    for 0 <= s <= pos_t.

One key vector per token is shared by all indexer heads. No further scale: any head or softmax
scale is taken as already folded into w. The causal range includes s = pos_t (the query's own
key).
"""
from __future__ import annotations

import numpy as np


def indexer_scores(q_idx, w, k_idx, kv, pos, bid) -> list:
    """Score rows, one fp64 array of length pos_t + 1 per query.

    q_idx [n_q, Hi, Di], w [n_q, Hi], k_idx [n_rows, Di] (any float dtype; widened to fp64),
    kv: a ContiguousKV / PagedKV row map, pos / bid [n_q].
    """
    q_idx = np.asarray(q_idx, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    k_idx = np.asarray(k_idx, dtype=np.float64)
    rows_out = []
    for t in range(q_idx.shape[0]):
        s = np.arange(int(pos[t]) + 1)
        keys = k_idx[kv.rows(int(bid[t]), s)]            # [L, Di]
        logits = q_idx[t] @ keys.T                         # [Hi, L]
        rows_out.append(w[t] @ np.maximum(logits, 0.0))    # [L]
    return rows_out
