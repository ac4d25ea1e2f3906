"""Pins for the all-gather + rerange oracle (no GPU)."""
import numpy as np
import pytest

from conftest import read_golden
from oracle import rerange as orr
from oracle import split as osplit


def test_worked_example_gathered_order():
    g = read_golden("rr_gathered_order_cp4.txt")
    sp, n = int(g[0][0].split()[1]), int(g[1][0].split()[1])
    x = np.arange(n)
    shards = [osplit.split_rows(x, sp, r) for r in range(sp)]
    gathered = orr.all_gather(shards)
    assert gathered.tolist() == [int(v) for v in g[2][1]]
    assert orr.rerange(gathered, n, sp).tolist() == [int(v) for v in g[3][1]]


def _brute(gathered, n, sp, stride):
    out = [None] * n
    row = 0
    for q in range(sp):
        start = q * stride if stride > 0 else row
        local = [g for g in range(n) if g % sp == q]
        for j, g in enumerate(local):
            out[g] = gathered[start + j].tolist()
        row = start + len(local)
    return out


@pytest.mark.parametrize("seed", range(10))
@pytest.mark.parametrize("padded", [False, True])
def test_rerange_inverts_gather_of_split(seed, padded):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(0, 60))
    sp = int(rng.integers(1, 9))
    x = rng.integers(0, 1 << 30, size=(n, 3))
    stride = (-(-n // sp) + int(rng.integers(0, 3))) if padded else 0
    shards = [osplit.split_rows(x, sp, r) for r in range(sp)]
    gathered = orr.all_gather(shards, stride)
    back = orr.rerange(gathered, n, sp, stride)
    assert np.array_equal(back, x)
    assert back.tolist() == _brute(gathered, n, sp, stride)


def test_padded_offsets():
    assert orr.rank_offsets(11, 4, 3).tolist() == [0, 3, 6, 9]
    assert orr.rank_offsets(11, 4, 0).tolist() == [0, 3, 6, 9]
    assert orr.rank_offsets(10, 4, 0).tolist() == [0, 3, 6, 8]
