"""Failure detection on the GPU without a fault: the bounded in-kernel wait gives up after its
limit and reports through the device error word; the context stays usable. The binding rejects
mis-shaped tensors before any launch (the C ABI takes bare pointers and cannot)."""
import numpy as np
import pytest
import torch

import workloads as W
from dsa_cases import Shard, dsa, i32

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports_timeout():
    m = dsa()
    m.dsa_read_device_errors()                      # start from a clean word
    m.dsa_selftest_bounded_wait(200_000)            # ~0.1 ms at GB300 clocks
    flags = m.dsa_read_device_errors()
    assert flags & m.DEVERR_TIMEOUT
    assert flags & 0xFF == 0xEE                     # the self-test's wait site
    assert flags & m.DEVERR_BAD_INDEX == 0          # the wait did not succeed
    # the context is still usable: a real call runs and is clean afterwards
    sh = Shard(W.WORKLOADS[0], 1)
    topk = sh.run_indexer_topk()
    torch.cuda.synchronize()
    assert topk.shape == (sh.n_q, sh.wl.topk)
    assert m.dsa_read_device_errors() == 0


def test_bounded_wait_limit_is_validated():
    m = dsa()
    with pytest.raises(m.DsaError):
        m.dsa_selftest_bounded_wait(0)


def test_binding_rejects_wrong_shapes_before_launch():
    m = dsa()
    sh = Shard(W.WORKLOADS[0], 1)
    ws = torch.empty(m.dsa_indexer_topk_workspace_size(sh.n_q, sh.max_ctx, sh.wl.topk),
                     dtype=torch.uint8, device="cuda")
    q_idx, w, k_idx = sh.idx.q_idx.cuda(), sh.idx.w.cuda(), sh.idx.k_idx.cuda()
    short = torch.empty((sh.n_q, sh.wl.topk - 1), dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):                 # topk narrower than k
        m.dsa_indexer_topk(q_idx, w, k_idx, sh.d_cu, sh.n_req, sh.d_pos, sh.d_bid, sh.wl.topk,
                           sh.max_ctx, short, ws)
    topk = torch.empty((sh.n_q, sh.wl.topk), dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):                 # pos with a row missing
        m.dsa_indexer_topk(q_idx, w, k_idx, sh.d_cu, sh.n_req, sh.d_pos[:-1], sh.d_bid,
                           sh.wl.topk, sh.max_ctx, topk, ws)
    with pytest.raises(ValueError):                 # w with the wrong head count
        m.dsa_indexer_topk(q_idx, w[:, :2].contiguous(), k_idx, sh.d_cu, sh.n_req, sh.d_pos,
                           sh.d_bid, sh.wl.topk, sh.max_ctx, topk, ws)
    o = torch.empty((sh.n_q, sh.wl.H, sh.wl.dv - 8), dtype=torch.bfloat16, device="cuda")
    q, c = sh.mla.q.cuda(), sh.mla.c.cuda()
    with pytest.raises(ValueError):                 # o narrower than q's head count / wrong lse
        m.dsa_sparse_mla(q, c, sh.d_cu, sh.n_req, sh.d_bid, topk, sh.wl.scale,
                         torch.empty((sh.n_q, 4, sh.wl.dv), dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(ValueError):
        m.dsa_sparse_mla(q, c, sh.d_cu, sh.n_req, sh.d_bid, topk, sh.wl.scale, o,
                         torch.empty((sh.n_q, 3), device="cuda"))
    cu = i32(W.cu_seqlens([10, 6]))
    with pytest.raises(ValueError):                 # pos shorter than the shard
        e = lambda n: torch.empty(n, dtype=torch.int32, device="cuda")
        m.dsa_rr_split_metadata(cu, 16, 4, 1, e(3), e(3), e(4))
    torch.cuda.synchronize()
    assert m.dsa_read_device_errors() == 0          # nothing was launched
