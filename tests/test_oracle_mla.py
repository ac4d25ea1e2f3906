"""Pins for the sparse / dense MLA oracle (no GPU)."""
import math

import numpy as np
import pytest
from scipy.special import logsumexp

from oracle import mla as omla
from oracle.kv import ContiguousKV, PagedKV


def _textbook(q, keys, vals, scale):
    """Softmax attention of one query row written out with plain loops."""
    logits = [scale * sum(q[d] * key[d] for d in range(len(q))) for key in keys]
    mx = max(logits)
    ex = [math.exp(x - mx) for x in logits]
    tot = sum(ex)
    out = [sum(ex[j] * vals[j][e] for j in range(len(keys))) / tot for e in range(len(vals[0]))]
    return out, mx + math.log(tot)


def test_single_head_full_value_is_textbook_attention():
    rng = np.random.default_rng(0)
    n, d = 12, 5
    q, c = rng.normal(size=(n, 1, d)), rng.normal(size=(n, d))
    pos = np.arange(n)
    o, lse = omla.dense_causal_mla(q, c, ContiguousKV([0, n]), pos, np.zeros(n, int), 0.7, d)
    for t in range(n):
        ref, l = _textbook(q[t, 0], c[:t + 1], c[:t + 1], 0.7)
        np.testing.assert_allclose(o[t, 0], ref, rtol=1e-12)
        assert abs(lse[t, 0] - l) < 1e-12


def test_one_selected_row_returns_its_value():
    rng = np.random.default_rng(1)
    q, c = rng.normal(size=(1, 3, 8)), rng.normal(size=(10, 8))
    o, lse = omla.sparse_mla(q, c, ContiguousKV([0, 10]), [0], np.array([[-1, 6, -1]]), 0.3, 4)
    assert np.array_equal(o[0], np.broadcast_to(c[6, :4], (3, 4)))
    np.testing.assert_allclose(lse[0], 0.3 * q[0] @ c[6], rtol=1e-14)


def test_lse_and_weights_against_library_routines():
    rng = np.random.default_rng(2)
    q, c = rng.normal(size=(2, 4, 9)), rng.normal(size=(30, 9))
    topk = np.array([[3, 7, 11, 29, -1], [0, 1, 2, 3, 4]])
    o, lse = omla.sparse_mla(q, c, ContiguousKV([0, 30]), [0, 0], topk, 0.25, 6)
    for t in range(2):
        sel = topk[t][topk[t] >= 0]
        S = 0.25 * q[t] @ c[sel].T
        np.testing.assert_allclose(lse[t], logsumexp(S, axis=1), rtol=1e-13)
        P = np.exp(S - logsumexp(S, axis=1, keepdims=True))
        np.testing.assert_allclose(o[t], P @ c[sel, :6], rtol=1e-12)


def test_order_of_selection_does_not_matter():
    rng = np.random.default_rng(3)
    q, c = rng.normal(size=(1, 4, 16)), rng.normal(size=(50, 16))
    sel = rng.choice(50, 20, replace=False)
    a = omla.sparse_mla(q, c, ContiguousKV([0, 50]), [0], sel[None], 0.2, 8)
    b = omla.sparse_mla(q, c, ContiguousKV([0, 50]), [0], np.sort(sel)[None], 0.2, 8)
    np.testing.assert_allclose(a[0], b[0], rtol=1e-13)
    np.testing.assert_allclose(a[1], b[1], rtol=1e-13)


@pytest.mark.parametrize("seed", range(4))
def test_topk_covering_context_equals_dense(seed):
    rng = np.random.default_rng(10 + seed)
    lengths = rng.integers(1, 30, 3)
    cu = np.concatenate([[0], np.cumsum(lengths)])
    N = int(cu[-1])
    bid = np.repeat(np.arange(3), lengths)
    pos = np.concatenate([np.arange(L) for L in lengths])
    q, c = rng.normal(size=(N, 2, 7)), rng.normal(size=(N, 7))
    k = 40
    topk = np.full((N, k), -1)
    for t in range(N):
        topk[t, :pos[t] + 1] = np.arange(pos[t] + 1)
    a = omla.sparse_mla(q, c, ContiguousKV(cu), bid, topk, 0.4, 5)
    b = omla.dense_causal_mla(q, c, ContiguousKV(cu), pos, bid, 0.4, 5)
    np.testing.assert_allclose(a[0], b[0], rtol=1e-13)
    np.testing.assert_allclose(a[1], b[1], rtol=1e-13)


def test_no_valid_entry_gives_zero_and_minus_inf():
    q, c = np.ones((1, 2, 3)), np.ones((4, 3))
    o, lse = omla.sparse_mla(q, c, ContiguousKV([0, 4]), [0], np.array([[-1, -1]]), 1.0, 2)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_paged_rows_follow_block_table():
    table = np.array([[2, 0], [1, 3]])
    kv = PagedKV(table, 4)
    assert kv.rows(0, np.array([0, 3, 4, 7])).tolist() == [8, 11, 0, 3]
    assert kv.rows(1, np.array([5])).tolist() == [13]
