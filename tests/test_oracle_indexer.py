"""Pins for the lightning-indexer oracle (no GPU)."""
import numpy as np
import pytest

from oracle import indexer as oidx
from oracle.kv import ContiguousKV, PagedKV
from oracle import split as osplit
from workloads import WORKLOADS, cu_seqlens, indexer_inputs, random_block_table


def _brute(q, w, k, cu, pos, bid):
    rows = []
    for t in range(len(pos)):
        row = []
        for s in range(int(pos[t]) + 1):
            acc = 0.0
            for h in range(q.shape[1]):
                d = 0.0
                for j in range(q.shape[2]):
                    d += float(q[t, h, j]) * float(k[cu[bid[t]] + s, j])
                acc += float(w[t, h]) * (d if d > 0 else 0.0)
            row.append(acc)
        rows.append(row)
    return rows


def _tiny(seed, integer):
    rng = np.random.default_rng(seed)
    lengths = rng.integers(1, 9, 3)
    cu = np.concatenate([[0], np.cumsum(lengths)])
    meta = osplit.round_robin_split(cu, 2, 1)
    n_q, Hi, Di = len(meta["pos"]), 3, 5
    if integer:
        q = rng.integers(-3, 4, (n_q, Hi, Di)).astype(float)
        k = rng.integers(-3, 4, (cu[-1], Di)).astype(float)
        w = rng.integers(-3, 4, (n_q, Hi)).astype(float)
    else:
        q, k, w = rng.normal(size=(n_q, Hi, Di)), rng.normal(size=(cu[-1], Di)), rng.normal(size=(n_q, Hi))
    return q, w, k, cu, meta["pos"], meta["bid"]


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_real(seed):
    q, w, k, cu, pos, bid = _tiny(seed, False)
    got = oidx.indexer_scores(q, w, k, ContiguousKV(cu), pos, bid)
    ref = _brute(q, w, k, cu, pos, bid)
    for a, b in zip(got, ref):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed", range(6))
def test_integer_inputs_exact(seed):
    q, w, k, cu, pos, bid = _tiny(seed, True)
    got = oidx.indexer_scores(q, w, k, ContiguousKV(cu), pos, bid)
    ref = _brute(q, w, k, cu, pos, bid)
    for a, b in zip(got, ref):
        assert a.tolist() == b                  # integers: exact equality
        assert np.all(a == np.round(a))


def test_single_head_unit_weight_is_relu_of_causal_dot():
    rng = np.random.default_rng(7)
    n = 17
    q = rng.normal(size=(n, 1, 6))
    k = rng.normal(size=(n, 6))
    w = np.ones((n, 1))
    pos = np.arange(n)
    got = oidx.indexer_scores(q, w, k, ContiguousKV([0, n]), pos, np.zeros(n, int))
    full = np.maximum(q[:, 0, :] @ k.T, 0.0)
    for t in range(n):
        np.testing.assert_allclose(got[t], full[t, :t + 1], rtol=1e-13)
    # non-negative dots: ReLU is the identity and the score is the plain causal q.k
    qp, kp = np.abs(q), np.abs(k)
    got = oidx.indexer_scores(qp, w, kp, ContiguousKV([0, n]), pos, np.zeros(n, int))
    for t in range(n):
        np.testing.assert_allclose(got[t], (qp[t, 0] @ kp[:t + 1].T), rtol=1e-13)


def test_one_hot_weight_selects_one_head():
    rng = np.random.default_rng(8)
    n, Hi, Di = 9, 4, 7
    q, k = rng.normal(size=(n, Hi, Di)), rng.normal(size=(n, Di))
    for h in range(Hi):
        w = np.zeros((n, Hi))
        w[:, h] = 2.5
        got = oidx.indexer_scores(q, w, k, ContiguousKV([0, n]), np.arange(n), np.zeros(n, int))
        for t in range(n):
            np.testing.assert_allclose(got[t], 2.5 * np.maximum(q[t, h] @ k[:t + 1].T, 0), rtol=1e-13)


def test_paged_layout_matches_contiguous():
    rng = np.random.default_rng(9)
    ctx = [70, 129, 5]
    page = 16
    table, total = random_block_table(ctx, page, 4)
    Di = 4
    logical = [rng.normal(size=(c, Di)) for c in ctx]
    pool = np.zeros((total * page, Di))
    for b, c in enumerate(ctx):
        for s in range(c):
            pool[table[b, s // page] * page + s % page] = logical[b][s]
    cu = np.concatenate([[0], np.cumsum(ctx)])
    flat = np.concatenate(logical)
    bid = np.array([0, 1, 1, 2])
    pos = np.array([69, 127, 128, 4])
    q, w = rng.normal(size=(4, 3, Di)), rng.normal(size=(4, 3))
    a = oidx.indexer_scores(q, w, pool, PagedKV(table, page), pos, bid)
    b = oidx.indexer_scores(q, w, flat, ContiguousKV(cu), pos, bid)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_tiny_workload_scores_are_exact_integers():
    wl = WORKLOADS[0]
    cu = cu_seqlens(wl.lengths)
    meta = osplit.round_robin_split(cu, wl.sp, 1)
    inp = indexer_inputs(wl, len(meta["pos"]), int(cu[-1]), 1)
    rows = oidx.indexer_scores(inp.q_idx.float().numpy(), inp.w.numpy(), inp.k_idx.float().numpy(),
                               ContiguousKV(cu), meta["pos"], meta["bid"])
    assert len(rows) == 64 and len(rows[-1]) == 254
    assert all(np.all(r == np.round(r)) and np.all(r >= 0) for r in rows)   # w >= 0 here
