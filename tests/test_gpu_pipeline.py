"""GPU end to end: the whole shard path in the launch configuration the benchmark times --
split metadata, each shard's rows gathered into the rank-major all-gather layout, rerange,
indexer + top-k, sparse MLA -- for every workload, checked on sampled queries against the
oracle. Integer-valued indexer inputs make the top-k index sets exact, so the MLA outputs are
compared against the oracle's own selection without feeding it anything from the GPU."""
import numpy as np
import pytest
import torch

import workloads as W
from dsa_cases import Shard, dsa, f64, gpu_split, i32, mla_close
from oracle import split as osplit

pytestmark = pytest.mark.gpu


def _rerange_kv(sh):
    """Split (row gather per shard) -> rank-major gathered buffer -> one rerange launch for
    k_idx and c together (the benchmark's dsa_rr_rerange_multi)."""
    m = dsa()
    wl, cu = sh.wl, sh.cu
    n = int(cu[-1])
    gathered, out = [], []
    for src in (sh.idx.k_idx.cuda(), sh.mla.c.cuda()):
        shards = [gpu_split(cu, wl.sp, r, src=src)["rows"] for r in range(wl.sp)]
        gathered.append(torch.cat(shards))
        out.append(torch.empty_like(src))
    m.dsa_rr_rerange_multi(gathered, out, n, wl.sp, 0)
    return out


def _run(sh, sel):
    m = dsa()
    wl = sh.wl
    if sh.block_table is None:
        g = gpu_split(sh.cu, wl.sp, sh.rank)
        assert np.array_equal(g["pos"], sh.pos) and np.array_equal(g["bid"], sh.bid)
        k_idx, c = _rerange_kv(sh)
        assert torch.equal(k_idx, sh.idx.k_idx.cuda()) and torch.equal(c, sh.mla.c.cuda())
    else:
        k_idx, c = sh.idx.k_idx.cuda(), sh.mla.c.cuda()
    ws = torch.empty(m.dsa_indexer_topk_workspace_size(sh.n_q, sh.max_ctx, wl.topk),
                     dtype=torch.uint8, device="cuda")
    topk = torch.full((sh.n_q, wl.topk), -9, dtype=torch.int32, device="cuda")
    m.dsa_indexer_topk(sh.idx.q_idx.cuda(), sh.idx.w.cuda(), k_idx, sh.d_cu, sh.n_req, sh.d_pos,
                       sh.d_bid, wl.topk, sh.max_ctx, topk, ws, block_table=sh.block_table)
    o = torch.full((sh.n_q, wl.H, wl.dv), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((sh.n_q, wl.H), float("nan"), device="cuda")
    mws = torch.empty(m.dsa_sparse_mla_workspace_size(sh.n_q), dtype=torch.uint8, device="cuda")
    m.dsa_sparse_mla_balanced(sh.mla.q.cuda(), c, sh.d_cu, sh.n_req, sh.d_bid, sh.d_pos, topk,
                              wl.scale, o, mws, lse=lse, block_table=sh.block_table)
    torch.cuda.synchronize()
    assert m.dsa_read_device_errors() == 0
    view = sh.oracle_view(sel)
    ref_topk = sh.oracle_topk(sh.oracle_scores(sel, view))
    got_topk = topk.cpu().numpy()[sel]
    assert np.array_equal(got_topk, ref_topk)
    ref_o, ref_lse = sh.oracle_mla(sel, ref_topk, view)
    mla_close(f64(o[torch.as_tensor(sel, device="cuda")]), ref_o)
    assert np.allclose(lse.cpu().numpy()[sel], ref_lse, atol=1e-3, rtol=1e-4)
    return o


def test_tiny_all_queries():
    sh = Shard(W.WORKLOADS[0], 1)
    _run(sh, np.arange(sh.n_q))


def test_varlen_rank3():
    sh = Shard(W.WORKLOADS[1], 3, integer_indexer=True)
    _run(sh, sh.samples(64))


@pytest.mark.parametrize("rank", [0, 7])
def test_long_prompt_shards(rank):
    sh = Shard(W.WORKLOADS[2], rank, integer_indexer=True)
    _run(sh, sh.samples(20, seed=rank))


@pytest.mark.parametrize("rank", [0, 1, 2, 3])
def test_many_request_shards(rank):
    sh = Shard(W.WORKLOADS[3], rank, integer_indexer=True)
    _run(sh, sh.samples(24, seed=rank))


def test_paged_decode():
    sh = Shard(W.WORKLOADS[4], 0, integer_indexer=True)
    _run(sh, sh.samples(16))


def test_round_robin_balance_of_many_request_batch():
    """Per-shard query counts differ by at most one and the causal work is balanced (the
    comparison the many-request workload asks for), while in-seq-split is not."""
    from oracle import inseq
    wl = W.WORKLOADS[3]
    cu = W.cu_seqlens(wl.lengths)
    rr = [osplit.round_robin_split(cu, wl.sp, r) for r in range(wl.sp)]
    counts = [len(m["pos"]) for m in rr]
    gpu_counts = [len(gpu_split(cu, wl.sp, r)["pos"]) for r in range(wl.sp)]
    assert gpu_counts == counts and max(counts) - min(counts) <= 1
    rr_pairs = [inseq.causal_pairs(m["pos"]) for m in rr]
    is_pairs = [inseq.causal_pairs(inseq.in_seq_split(wl.lengths, wl.sp, r)[1]) for r in range(wl.sp)]
    spread = lambda x: (max(x) - min(x)) / np.mean(x)
    assert spread(rr_pairs) < 1e-3 and spread(is_pairs) > 0.5
