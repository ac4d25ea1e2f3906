"""Pins for the top-k oracle (no GPU)."""
import numpy as np
import pytest

from oracle.topk import topk_indices


def _rank_rule(scores, k):
    """Index i is chosen iff fewer than k entries beat it: larger score, or equal and lower index."""
    chosen = []
    for i in range(len(scores)):
        beat = sum(1 for j in range(len(scores))
                   if scores[j] > scores[i] or (scores[j] == scores[i] and j < i))
        if beat < k:
            chosen.append(i)
    return chosen + [-1] * (k - len(chosen))


@pytest.mark.parametrize("seed", range(20))
def test_rank_rule_brute_force(seed):
    rng = np.random.default_rng(seed)
    L = int(rng.integers(1, 80))
    k = int(rng.integers(1, 40))
    scores = rng.integers(-4, 5, L).astype(np.float64)       # heavy ties
    assert topk_indices(scores, k).tolist() == _rank_rule(scores, k)


@pytest.mark.parametrize("seed", range(10))
def test_properties_real(seed):
    rng = np.random.default_rng(50 + seed)
    L, k = int(rng.integers(40, 400)), int(rng.integers(1, 40))
    s = np.round(rng.normal(size=L), 1)
    out = topk_indices(s, k)
    sel = out[out >= 0]
    rest = np.setdiff1d(np.arange(L), sel)
    assert len(sel) == min(k, L) and np.all(np.diff(sel) > 0)
    assert s[sel].min() >= s[rest].max()
    thr = s[sel].min()
    ties = np.flatnonzero(s == thr)
    chosen_ties = np.intersect1d(ties, sel)
    assert np.array_equal(chosen_ties, ties[:len(chosen_ties)])   # lowest-index prefix of ties


def test_short_row_takes_all_and_pads():
    assert topk_indices(np.array([3.0, 1.0, 2.0]), 5).tolist() == [0, 1, 2, -1, -1]
    assert topk_indices(np.array([]), 2).tolist() == [-1, -1]


def test_negative_zero_equals_zero():
    s = np.array([-0.0, 0.0, -0.0, -1.0, 0.0])
    assert topk_indices(s, 2).tolist() == [0, 1]
    s32 = np.array([-0.0, 0.0, -0.0, -1.0], dtype=np.float32)
    assert topk_indices(s32, 3).tolist() == [0, 1, 2]


def test_all_equal_takes_lowest_indices():
    assert topk_indices(np.full(100, 7.0), 32).tolist() == list(range(32))
