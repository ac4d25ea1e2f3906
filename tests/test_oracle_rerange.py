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


def test_rerange_into_pages_hand_example():
    # 6 tokens (values 0..5), requests of 4 and 2 tokens, sp = 2 (gathered T0,T2,T4,T1,T3,T5),
    # pages of 2 rows; request 0 uses pages 3 then 0, request 1 uses page 1. By hand: tokens 0,1
    # -> rows 6,7; tokens 2,3 -> rows 0,1; tokens 4,5 -> rows 2,3; rows 4,5 untouched (-1).
    gathered = np.array([0, 2, 4, 1, 3, 5])
    pool = np.full(8, -1)
    out = orr.rerange_into_pages(gathered, [0, 4, 6], 2, 0, [[3, 0], [1, -1]], 2, pool)
    assert out.tolist() == [2, 3, 4, 5, -1, -1, 0, 1]


@pytest.mark.parametrize("seed", range(6))
def test_rerange_into_pages_contiguous_pages_is_the_rerange(seed):
    # request lengths that are whole pages and a block table of consecutive pages in request
    # order: the pool is exactly the logical buffer
    rng = np.random.default_rng(seed)
    ps, sp = int(rng.choice([2, 4, 8])), int(rng.integers(1, 6))
    pages = rng.integers(1, 4, size=int(rng.integers(1, 5)))
    cu = np.concatenate([[0], np.cumsum(pages * ps)])
    n = int(cu[-1])
    table = np.full((len(pages), int(pages.max())), -1)
    at = 0
    for b, p in enumerate(pages):
        table[b, :p] = np.arange(at, at + p)
        at += p
    x = rng.integers(0, 1 << 30, size=(n, 3))
    gathered = orr.all_gather([osplit.split_rows(x, sp, r) for r in range(sp)])
    out = orr.rerange_into_pages(gathered, cu, sp, 0, table, ps, np.zeros_like(x))
    assert np.array_equal(out, x)


@pytest.mark.parametrize("seed", range(6))
def test_rerange_into_pages_reads_back_through_the_page_map(seed):
    from oracle.kv import PagedKV
    rng = np.random.default_rng(100 + seed)
    ps, sp = int(rng.choice([2, 3, 64])), int(rng.integers(1, 9))
    lengths = rng.integers(0, 200, size=int(rng.integers(1, 6)))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    need = [-(-int(L) // ps) for L in lengths]
    perm = rng.permutation(sum(need) + 3)             # a few spare pages stay untouched
    table = np.full((len(lengths), max(max(need), 1)), -1)
    at = 0
    for b, p in enumerate(need):
        table[b, :p] = perm[at:at + p]
        at += p
    n = int(cu[-1])
    x = rng.integers(0, 1 << 30, size=(n, 2))
    stride = -(-n // sp) + 1
    gathered = orr.all_gather([osplit.split_rows(x, sp, r) for r in range(sp)], stride)
    pool0 = np.full(((sum(need) + 3) * ps, 2), -7)
    pool = orr.rerange_into_pages(gathered, cu, sp, stride, table, ps, pool0)
    kv = PagedKV(table, ps)
    for b in range(len(lengths)):
        s = np.arange(lengths[b])
        assert np.array_equal(pool[kv.rows(b, s)], x[cu[b] + s])
    written = np.zeros(len(pool), bool)
    for b in range(len(lengths)):
        written[kv.rows(b, np.arange(lengths[b]))] = True
    assert (pool[~written] == -7).all()


def test_local_cache_worked_example():
    # CP = 4, one request [T0 .. T7]: each rank's cache keeps exactly the tokens the page names
    # for it (rank 1: K1 then K5). Pages of 2 rows; every rank's request uses its page 5.
    g = read_golden("local_cache_cp4.txt")
    sp, n = int(g[0][0].split()[1]), int(g[1][0].split()[1])
    x = np.arange(n) * 10                                  # K_g = 10 g
    for key, vals in g[2:]:
        r = int(key.split()[1])
        local = osplit.split_rows(x, sp, r)
        pool = orr.cache_local_into_pages(local, [0, n], sp, r, [[5]], 2, np.full(12, -1))
        assert pool[10:12].tolist() == [10 * int(v) for v in vals]
        assert (pool[:10] == -1).all()


def test_local_cache_one_shard_is_the_paged_rerange():
    # sp = 1: the rank owns every token, so its cache is the full paged write of the batch
    rng = np.random.default_rng(5)
    lengths = [7, 3, 12]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    ps = 4
    need = [-(-L // ps) for L in lengths]
    perm = rng.permutation(sum(need))
    table = np.full((3, max(need)), -1)
    at = 0
    for b, p in enumerate(need):
        table[b, :p] = perm[at:at + p]
        at += p
    x = rng.integers(0, 1 << 30, size=(int(cu[-1]), 2))
    pool0 = np.zeros((sum(need) * ps, 2), dtype=x.dtype)
    a = orr.cache_local_into_pages(x, cu, 1, 0, table, ps, pool0)
    b = orr.rerange_into_pages(x, cu, 1, 0, table, ps, pool0)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("seed", range(6))
def test_local_caches_partition_the_batch(seed):
    # Every logical token lands in exactly one rank's cache, at its index among the request's
    # tokens on that rank; read back through each rank's page map it is the split's row.
    from oracle.kv import PagedKV
    rng = np.random.default_rng(200 + seed)
    sp, ps = int(rng.integers(1, 9)), int(rng.choice([1, 3, 64]))
    lengths = rng.integers(0, 150, size=int(rng.integers(1, 6)))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    n = int(cu[-1])
    x = rng.integers(0, 1 << 30, size=(n, 2))
    seen = np.zeros(n, dtype=np.int64)
    for r in range(sp):
        tokens = osplit.shard_tokens(n, sp, r)
        counts = [int(np.sum((tokens >= cu[b]) & (tokens < cu[b + 1]))) for b in range(len(lengths))]
        need = [-(-c // ps) for c in counts]
        perm = rng.permutation(sum(need) + 2)
        table = np.full((len(lengths), max(max(need), 1)), -1)
        at = 0
        for b, p in enumerate(need):
            table[b, :p] = perm[at:at + p]
            at += p
        pool = orr.cache_local_into_pages(osplit.split_rows(x, sp, r), cu, sp, r, table, ps,
                                          np.full(((sum(need) + 2) * ps, 2), -7))
        kv = PagedKV(table, ps)
        for b in range(len(lengths)):
            mine = tokens[(tokens >= cu[b]) & (tokens < cu[b + 1])]
            assert np.array_equal(pool[kv.rows(b, np.arange(len(mine)))], x[mine])
            assert np.all(mine % sp == r)
            seen[mine] += 1
    assert (seen == 1).all()
