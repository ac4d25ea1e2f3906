"""Pins for the round-robin split oracle (no GPU)."""
import numpy as np
import pytest

from conftest import read_golden
from oracle import split as osplit
from oracle.inseq import causal_pairs
from workloads import WORKLOADS, cu_seqlens, random_lengths


def test_worked_example_8_tokens_cp4():
    g = read_golden("rr_split_cp4_8tokens.txt")
    sp = int(g[0][0].split()[1])
    n = int(g[1][0].split()[1])
    for key, vals in g[2:]:
        r = int(key.split()[1])
        meta = osplit.round_robin_split([0, n], sp, r)
        assert meta["gidx"].tolist() == [int(v) for v in vals]
        assert meta["pos"].tolist() == [int(v) for v in vals]     # one request: pos == g
        assert meta["bid"].tolist() == [0] * len(vals)
        assert meta["cu_shard"].tolist() == [0, len(vals)]


def test_rank1_queries_and_causal_ranges():
    g = dict(read_golden("rank1_attention_cp4.txt")[3:])
    meta = osplit.round_robin_split([0, 8], 4, 1)
    assert meta["gidx"].tolist() == [int(v) for v in g["queries"]]
    for t, p in enumerate(meta["pos"]):
        assert list(range(int(p) + 1)) == [int(v) for v in g[f"keys_seen_by_{int(meta['gidx'][t])}"]]


def _brute(cu, sp, r):
    gidx, bid, pos = [], [], []
    n = cu[-1]
    for g in range(n):
        if g % sp != r:
            continue
        b = 0
        while not (cu[b] <= g < cu[b + 1]):
            b += 1
        gidx.append(g)
        bid.append(b)
        pos.append(g - cu[b])
    cu_shard = [0]
    for b in range(len(cu) - 1):
        cu_shard.append(cu_shard[-1] + sum(1 for x in bid if x == b))
    return gidx, bid, pos, cu_shard


@pytest.mark.parametrize("seed", range(12))
def test_brute_force_random_batches(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 7))
    lengths = rng.integers(0, 23, B)          # includes empty requests
    cu = [0] + np.cumsum(lengths).tolist()
    sp = int(rng.integers(1, 9))
    for r in range(sp):
        meta = osplit.round_robin_split(cu, sp, r)
        gidx, bid, pos, cu_shard = _brute(cu, sp, r)
        assert meta["gidx"].tolist() == gidx
        assert meta["bid"].tolist() == bid
        assert meta["pos"].tolist() == pos
        assert meta["cu_shard"].tolist() == cu_shard


@pytest.mark.parametrize("seed", range(8))
def test_shard_cu_closed_form_and_balance(seed):
    rng = np.random.default_rng(100 + seed)
    lengths = rng.integers(0, 5000, int(rng.integers(1, 40)))
    cu = cu_seqlens(lengths)
    n = int(cu[-1])
    sp = int(rng.integers(1, 17))
    counts, seen = [], np.zeros(n, dtype=np.int64)
    for r in range(sp):
        meta = osplit.round_robin_split(cu, sp, r)
        # closed form: tokens g < X with g = r (mod sp) number max(0, ceil((X - r) / sp))
        closed = [max(0, -(-(int(x) - r) // sp)) for x in cu]
        assert meta["cu_shard"].tolist() == closed
        counts.append(len(meta["gidx"]))
        seen[meta["gidx"]] += 1
    # balance stated on the page: per-rank token counts differ by at most one, any batch
    assert max(counts) - min(counts) <= 1
    assert sum(counts) == n and np.all(seen == 1)        # the shards partition 0..N-1


def test_varlen_workload_rank3_counts():
    wl = WORKLOADS[1]
    meta = osplit.round_robin_split(cu_seqlens(wl.lengths), wl.sp, 3)
    per_req = np.diff(meta["cu_shard"]).tolist()
    assert per_req == [1000, 100, 1, 375] and len(meta["gidx"]) == 1476


def test_many_request_round_robin_is_balanced():
    wl = WORKLOADS[3]
    cu = cu_seqlens(wl.lengths)
    assert int(cu[-1]) == 71014
    pairs = [causal_pairs(osplit.round_robin_split(cu, wl.sp, r)["pos"]) for r in range(wl.sp)]
    assert (max(pairs) - min(pairs)) / np.mean(pairs) < 1e-3


def test_split_rows_gathers_rows():
    x = np.arange(30).reshape(10, 3)
    assert osplit.split_rows(x, 4, 2).tolist() == [[6, 7, 8], [18, 19, 20]]


def test_random_lengths_generator_is_seeded():
    assert random_lengths(5, 1, 9, 3) == random_lengths(5, 1, 9, 3)


def test_decode_split_positions_continue_the_context():
    # two requests with contexts of 10 and 5 tokens before this step, 2 and 3 new tokens;
    # sp = 2: flattened new tokens 0..4 -> rank 0 gets 0, 2, 4; rank 1 gets 1, 3.
    # request 0's new tokens sit at positions 10, 11; request 1's at 5, 6, 7.
    r0 = osplit.round_robin_split_decode([0, 2, 5], [10, 5], 2, 0)
    r1 = osplit.round_robin_split_decode([0, 2, 5], [10, 5], 2, 1)
    assert r0["bid"].tolist() == [0, 1, 1] and r0["pos"].tolist() == [10, 5, 7]
    assert r1["bid"].tolist() == [0, 1] and r1["pos"].tolist() == [11, 6]
    assert r0["cu_shard"].tolist() == [0, 1, 3] and r1["cu_shard"].tolist() == [0, 1, 2]


def test_decode_split_with_one_shard_is_the_decode_batch():
    # sp = 1 keeps every new token: the positions are the last q tokens of each context, the
    # layout of the decode workload (its queries at C - 2 and C - 1)
    import workloads as W
    wl = W.WORKLOADS[4]
    q = wl.decode_queries
    ctx = np.asarray(wl.lengths, dtype=np.int64)
    cu_new = np.arange(len(ctx) + 1, dtype=np.int64) * q
    out = osplit.round_robin_split_decode(cu_new, ctx - q, 1, 0)
    bid, pos = W.decode_queries(wl.lengths, q)
    assert np.array_equal(out["bid"], bid) and np.array_equal(out["pos"], pos)


@pytest.mark.parametrize("seed", range(5))
def test_decode_split_zero_base_is_the_prefill_split(seed):
    rng = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(rng.integers(0, 5, int(rng.integers(1, 9))))])
    sp = int(rng.integers(1, 6))
    for r in range(sp):
        a = osplit.round_robin_split(cu, sp, r)
        b = osplit.round_robin_split_decode(cu, np.zeros(len(cu) - 1), sp, r)
        for k in a:
            assert np.array_equal(a[k], b[k])
