"""GPU parity: tensor-core lightning-indexer scores and the top-k built on them vs the oracle.

Integer-valued inputs make every score an exact fp32 integer, so scores and index sets are
compared bit for bit. bf16 N(0,1) inputs are compared against a derived fp32 rounding bound,
and index sets may differ only at near-ties of the k-th score."""
import numpy as np
import pytest
import torch

import workloads as W
from dsa_cases import Shard, check_topk_near_ties, score_error_bound

pytestmark = pytest.mark.gpu


def _exact_check(sh, sel):
    scores, topk = sh.run_indexer()
    view = sh.oracle_view(sel)
    ora = sh.oracle_scores(sel, view)
    ora_topk = sh.oracle_topk(ora)
    s_np = scores.cpu().numpy()
    t_np = topk.cpu().numpy()
    for i, t in enumerate(sel):
        L = int(sh.pos[t]) + 1
        assert np.array_equal(s_np[t, :L].astype(np.float64), ora[i]), (t, L)
        assert np.array_equal(t_np[t], ora_topk[i]), t
    return topk


def test_tiny_workload_all_queries_exact():
    sh = Shard(W.WORKLOADS[0], 1)
    _exact_check(sh, np.arange(sh.n_q))


def test_varlen_integer_inputs_exact():
    sh = Shard(W.WORKLOADS[1], 3, integer_indexer=True)
    _exact_check(sh, sh.samples(160))


@pytest.mark.parametrize("wid,rank", [(2, 5), (3, 2)])
def test_long_and_many_request_shards_integer_exact(wid, rank):
    sh = Shard(W.WORKLOADS[wid], rank, integer_indexer=True)
    _exact_check(sh, sh.samples(48))


def test_paged_decode_integer_exact():
    sh = Shard(W.WORKLOADS[4], 0, integer_indexer=True)
    _exact_check(sh, sh.samples(24))


def test_varlen_bf16_normal_within_bound_and_near_ties():
    wl = W.WORKLOADS[1]
    sh = Shard(wl, 3)
    scores, topk = sh.run_indexer()
    sel = sh.samples(96)
    view = sh.oracle_view(sel)
    ora = sh.oracle_scores(sel, view)
    s_np, t_np = scores.cpu().numpy(), topk.cpu().numpy()
    swaps = 0
    for i, t in enumerate(sel):
        L = int(sh.pos[t]) + 1
        bound = score_error_bound(view, i, L, wl.Di, wl.Hi)
        err = np.abs(s_np[t, :L].astype(np.float64) - ora[i])
        assert np.all(err <= bound), (t, float(np.max(err / bound)))
        swaps += check_topk_near_ties(t_np[t], sh.oracle_topk([ora[i]])[0], ora[i], wl.topk)
    assert swaps <= len(sel)          # near-tie swaps are rare; report through the assert


def test_composite_call_equals_separate_calls():
    sh = Shard(W.WORKLOADS[1], 3, integer_indexer=True)
    _, topk = sh.run_indexer()
    assert torch.equal(sh.run_indexer_topk(), topk)


@pytest.mark.parametrize("k", [700, 3000, 8000])
def test_groups_whose_histories_fit_in_k_are_left_out(k):
    """dsa_indexer_topk computes no score for a group of queries whose histories all hold at most
    k keys (the top-k of such a query is every key, whatever the scores): with k = 700, 3,000 or
    8,000 on the varlen shard (histories of up to 8,000 keys) a few, most or all groups are left
    out, and the index sets still equal the oracle's (integer inputs)."""
    from oracle.topk import topk_rows
    sh = Shard(W.WORKLOADS[1], 3, integer_indexer=True)
    t_np = sh.run_indexer_topk(k=k).cpu().numpy()
    for t in np.flatnonzero(sh.pos + 1 <= k):
        L = int(sh.pos[t]) + 1
        assert np.array_equal(t_np[t, :L], np.arange(L)) and np.all(t_np[t, L:] == -1), t
    near = np.argsort(np.abs(sh.pos.astype(np.int64) + 1 - k), kind="stable")[:6]
    sel = np.union1d(sh.samples(40), near)            # the queries on either side of k as well
    ref = topk_rows(sh.oracle_scores(sel), k)
    for i, t in enumerate(sel):
        assert np.array_equal(t_np[t], ref[i]), (t, int(sh.pos[t]))


def test_row_longer_than_max_ctx_is_flagged_not_written():
    import deepseek_v3_sparse_round_gb300 as dsa
    sh = Shard(W.WORKLOADS[0], 1)
    dsa.dsa_read_device_errors()
    sh.max_ctx = 100                       # queries at pos >= 100 violate the stated maximum
    scores, topk = sh.run_indexer()
    flags = dsa.dsa_read_device_errors()
    assert flags & (dsa.DEVERR_BAD_INDEX | dsa.DEVERR_BAD_LENGTH)
    assert not torch.isnan(scores[:, :100][torch.as_tensor(sh.pos < 100)]).all()


# ---- the fused path: dsa_indexer_topk with max_ctx > 8192 has the indexer histogram each
# score's first radix digit, and the top-k reads each row once, keeping only candidates. It
# must give exactly the index sets of the separate calls (same scores, same selection rule).
def _fused_equals_separate(sh, max_ctx=None):
    if max_ctx is not None:
        sh.max_ctx = max_ctx
    assert sh.max_ctx > 8192
    _, sep = sh.run_indexer()
    fused = sh.run_indexer_topk()
    torch.cuda.synchronize()
    assert torch.equal(fused, sep)
    import deepseek_v3_sparse_round_gb300 as dsa
    assert dsa.dsa_read_device_errors() == 0
    return fused


@pytest.mark.parametrize("wid,rank,integer", [(2, 5, True), (2, 1, False), (4, 0, True),
                                              (4, 0, False)])
def test_fused_indexer_topk_long_rows(wid, rank, integer):
    sh = Shard(W.WORKLOADS[wid], rank, integer_indexer=integer)
    fused = _fused_equals_separate(sh).cpu().numpy()
    if integer:                                       # exact scores: the oracle's sets, bit for bit
        sel = sh.samples(24)
        ora = sh.oracle_topk(sh.oracle_scores(sel))
        for i, t in enumerate(sel):
            assert np.array_equal(fused[t], ora[i]), t


@pytest.mark.parametrize("wid,rank", [(0, 1), (1, 3), (3, 2)])
def test_fused_path_on_short_rows(wid, rank):
    """The fused path forced on workloads whose rows are short (a larger max_ctx is a valid
    upper bound): heavy integer ties (workload 0), rows around k, every request length."""
    sh = Shard(W.WORKLOADS[wid], rank, integer_indexer=True)
    fused = _fused_equals_separate(sh, max_ctx=9000).cpu().numpy()
    sel = sh.samples(32)
    ora = sh.oracle_topk(sh.oracle_scores(sel))
    for i, t in enumerate(sel):
        assert np.array_equal(fused[t], ora[i]), t


def test_fused_crowded_boundary_bin_takes_the_global_path():
    """All scores equal (q_idx = 0): the boundary bin holds the whole row, more entries than the
    shared-memory list takes, so rows over 8,192 keys go through the global-memory passes; the
    result is still the lowest k indices."""
    sh = Shard(W.WORKLOADS[2], 7, integer_indexer=True)
    sh.idx.q_idx = torch.zeros_like(sh.idx.q_idx)
    fused = _fused_equals_separate(sh).cpu().numpy()
    for t in (0, 2047, 2048, 4095):
        L = int(sh.pos[t]) + 1
        want = np.full(2048, -1)
        want[:min(L, 2048)] = np.arange(min(L, 2048))
        assert np.array_equal(fused[t], want), t


def test_fused_misleading_sample_stays_exact():
    """The indexer's histogram samples one key position in 16. Keys at sampled positions are
    made to score higher than the rest (their k_idx rows tripled), so the sample points at a
    threshold that keeps fewer than k entries of a long row: the kernel notices from the exact
    count and takes the global-memory passes. The index sets are still the oracle's."""
    sh = Shard(W.WORKLOADS[2], 3, integer_indexer=True)
    k = sh.idx.k_idx.clone()
    k[0::16] = (k[0::16].float() * 3).to(torch.bfloat16)         # one request: row = position
    sh.idx.k_idx = k
    fused = _fused_equals_separate(sh).cpu().numpy()
    sel = np.array([4095, 4000, 2600, 1500, 1100])
    ora = sh.oracle_topk(sh.oracle_scores(sel))
    for i, t in enumerate(sel):
        assert np.array_equal(fused[t], ora[i]), t
