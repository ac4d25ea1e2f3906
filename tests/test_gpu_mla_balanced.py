"""GPU: sparse MLA with the pairs' work ordered by each query's estimated size. The schedule only
changes which CTA pair runs which query, so o and lse must equal the plain call's bit for bit;
a sample is also checked against the fp64 oracle on its own."""
import numpy as np
import pytest
import torch

import workloads as W
from dsa_cases import Shard, dsa, f64, i32, mla_close

pytestmark = pytest.mark.gpu


def _both(sh, topk, pos):
    m = dsa()
    q, c = sh.mla.q.cuda(), sh.mla.c.cuda()
    shape_o, shape_l = (sh.n_q, sh.wl.H, sh.wl.dv), (sh.n_q, sh.wl.H)
    o1 = torch.full(shape_o, float("nan"), dtype=torch.bfloat16, device="cuda")
    l1 = torch.full(shape_l, float("nan"), device="cuda")
    o2, l2 = o1.clone(), l1.clone()
    m.dsa_sparse_mla(q, c, sh.d_cu, sh.n_req, sh.d_bid, topk, sh.wl.scale, o1, l1,
                     block_table=sh.block_table)
    ws = torch.empty(m.dsa_sparse_mla_workspace_size(sh.n_q), dtype=torch.uint8, device="cuda")
    ws.fill_(0xAB)                                   # the schedule must not read stale contents
    m.dsa_sparse_mla_balanced(q, c, sh.d_cu, sh.n_req, sh.d_bid, pos, topk, sh.wl.scale, o2, ws,
                              lse=l2, block_table=sh.block_table)
    torch.cuda.synchronize()
    assert m.dsa_read_device_errors() == 0
    return (o1, l1), (o2, l2)


@pytest.mark.parametrize("wid,rank", [(1, 3), (3, 0), (4, 0)])
def test_balanced_equals_plain_on_whole_shards(wid, rank):
    sh = Shard(W.WORKLOADS[wid], rank, integer_indexer=False)
    topk = sh.run_indexer_topk()
    (o1, l1), (o2, l2) = _both(sh, topk, sh.d_pos)
    assert torch.equal(o1, o2)
    assert torch.equal(l1, l2)


def test_balanced_with_positions_unrelated_to_the_work():
    # Beyond bounding the valid entries (an entry must not exceed its query's position), pos
    # only steers the schedule: positions at or above each query's own, raised by random
    # amounts (past k, shuffled in size), keep every entry valid and change nothing.
    sh = Shard(W.WORKLOADS[1], 3, integer_indexer=False)
    topk = sh.run_indexer_topk()
    rng = np.random.default_rng(5)
    pos = (sh.pos.astype(np.int64) + rng.integers(0, 20000, sh.n_q)).astype(np.int32)
    (o1, l1), (o2, l2) = _both(sh, topk, i32(pos))
    assert torch.equal(o1, o2)
    assert torch.equal(l1, l2)


def test_balanced_sample_matches_oracle():
    sh = Shard(W.WORKLOADS[1], 3, integer_indexer=False)
    sel = sh.samples(24)
    view = sh.oracle_view(sel)
    topk_np = sh.oracle_topk(sh.oracle_scores(sel, view))
    full = np.full((sh.n_q, sh.wl.topk), -1, dtype=np.int32)
    full[sel] = topk_np
    (_, _), (o2, l2) = _both(sh, i32(full), sh.d_pos)
    ref_o, ref_lse = sh.oracle_mla(sel, topk_np, view)
    mla_close(f64(o2[torch.as_tensor(sel, device="cuda")]), ref_o)
    assert np.allclose(l2[torch.as_tensor(sel, device="cuda")].cpu().numpy(), ref_lse,
                       atol=1e-3, rtol=1e-4)


def test_short_workspace_and_missing_pos_rejected():
    m = dsa()
    sh = Shard(W.WORKLOADS[0], 1)
    topk = torch.full((sh.n_q, sh.wl.topk), -1, dtype=torch.int32, device="cuda")
    q, c = sh.mla.q.cuda(), sh.mla.c.cuda()
    o = torch.empty((sh.n_q, sh.wl.H, sh.wl.dv), dtype=torch.bfloat16, device="cuda")
    small = torch.empty(4, dtype=torch.uint8, device="cuda")
    # the small-head path runs unscheduled; the 128-head workspace checks run on the host
    m.dsa_sparse_mla_balanced(q, c, sh.d_cu, sh.n_req, sh.d_bid, sh.d_pos, topk, sh.wl.scale, o,
                              torch.empty(m.dsa_sparse_mla_workspace_size(sh.n_q),
                                          dtype=torch.uint8, device="cuda"))
    with pytest.raises(m.DsaError):
        m.dsa_sparse_mla_balanced(q, c, sh.d_cu, sh.n_req, sh.d_bid, sh.d_pos, topk, sh.wl.scale,
                                  o, small)
    with pytest.raises(ValueError):
        m.dsa_sparse_mla_balanced(q, c, sh.d_cu, sh.n_req, sh.d_bid, sh.d_pos, topk, sh.wl.scale,
                                  o, None)
    assert m.dsa_sparse_mla_workspace_size(0) == 0
    assert m.dsa_sparse_mla_workspace_size(1476) == 1476 * 4


@pytest.mark.parametrize("n", [1, 2, 75, 77, 153])
def test_query_counts_around_the_number_of_pairs(n):
    """Fewer queries than CTA pairs (1, 2), one below and one above a pair per query on a 152-SM
    GPU (75, 77: 76 pairs), and two queries per pair plus one (153): plain and balanced calls on
    the same subset agree bit for bit and match the oracle."""
    m = dsa()
    sh = Shard(W.WORKLOADS[1], 3, integer_indexer=False)
    sel = np.linspace(0, sh.n_q - 1, n).round().astype(np.int64)
    view = sh.oracle_view(sel)
    topk_np = sh.oracle_topk(sh.oracle_scores(sel, view))
    sel_t = torch.as_tensor(sel, device="cuda")
    q, c, topk = sh.mla.q[sel_t].cuda(), sh.mla.c.cuda(), i32(topk_np)
    bid, pos = i32(sh.bid[sel]), i32(sh.pos[sel])
    o1 = torch.full((n, sh.wl.H, sh.wl.dv), float("nan"), dtype=torch.bfloat16, device="cuda")
    l1 = torch.full((n, sh.wl.H), float("nan"), device="cuda")
    o2, l2 = o1.clone(), l1.clone()
    m.dsa_sparse_mla(q, c, sh.d_cu, sh.n_req, bid, topk, sh.wl.scale, o1, l1)
    ws = torch.empty(m.dsa_sparse_mla_workspace_size(n), dtype=torch.uint8, device="cuda")
    m.dsa_sparse_mla_balanced(q, c, sh.d_cu, sh.n_req, bid, pos, topk, sh.wl.scale, o2, ws, lse=l2)
    torch.cuda.synchronize()
    assert m.dsa_read_device_errors() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    ref_o, ref_lse = sh.oracle_mla(sel, topk_np, view)
    mla_close(f64(o1), ref_o)
    assert np.allclose(l1.cpu().numpy(), ref_lse, atol=1e-3, rtol=1e-4)
