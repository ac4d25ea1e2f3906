"""Oracle: sparse MLA over each query's selected latent rows, and dense causal MLA.

Test infrastructure only (see the package docstring).

"[RFC]: Parallel strategy for Deepseek v3.2 like models": in sparse MLA each query attends only
the top-k keys the indexer chose, with all heads ("full head on mla part"). Definition (MLA in
its absorbed form, one shared latent row per token):

    S[h, j] = scale * sum_d q[t, h, d] * c[row(b_t, idx_j), d]     over d < dqk
    P[h, :] = softmax_j(S[h, :])
    o[t, h, :] = sum_j P[h, j] * c[row(b_t, idx_j), :dv]
    lse[t, h] = log sum_j exp(S[h, j])

over the valid selected entries idx_j >= 0 (-1 entries are padding). V is the first dv columns
of the same latent row. A query with no valid entry gets o = 0 and lse = -inf. The softmax is
the max-subtracted form, in fp64.
"""
from __future__ import annotations

import numpy as np


def _attend(qt, keys, scale, dv):
    S = scale * (qt @ keys.T)                       # [H, m]
    m = S.max(axis=1, keepdims=True)
    E = np.exp(S - m)
    l = E.sum(axis=1, keepdims=True)
    o = (E @ keys[:, :dv]) / l
    lse = (m + np.log(l))[:, 0]
    return o, lse


def sparse_mla(q, c, kv, bid, topk, scale: float, dv: int):
    """q [n_q, H, dqk], c [n_rows, dqk], topk [n_q, k] (entries >= 0 valid) -> (o, lse)."""
    q = np.asarray(q, dtype=np.float64)
    c = np.asarray(c, dtype=np.float64)
    n_q, H = q.shape[0], q.shape[1]
    o = np.zeros((n_q, H, dv))
    lse = np.full((n_q, H), -np.inf)
    for t in range(n_q):
        sel = np.asarray(topk[t])
        sel = sel[sel >= 0]
        if sel.shape[0] == 0:
            continue
        keys = c[kv.rows(int(bid[t]), sel)]
        o[t], lse[t] = _attend(q[t], keys, scale, dv)
    return o, lse


def dense_causal_mla(q, c, kv, pos, bid, scale: float, dv: int):
    """The same attention over every key s <= pos_t of the query's request."""
    q = np.asarray(q, dtype=np.float64)
    c = np.asarray(c, dtype=np.float64)
    n_q, H = q.shape[0], q.shape[1]
    o = np.zeros((n_q, H, dv))
    lse = np.full((n_q, H), -np.inf)
    for t in range(n_q):
        keys = c[kv.rows(int(bid[t]), np.arange(int(pos[t]) + 1))]
        o[t], lse[t] = _attend(q[t], keys, scale, dv)
    return o, lse
