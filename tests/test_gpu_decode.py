"""GPU: round-robin sharding of a decode step's new tokens. The decode split metadata is
bit-exact against the oracle; a decode shard runs indexer + top-k and sparse MLA on the paged
KV from that metadata and matches the oracle on every one of its queries (integer indexer
inputs, so the index sets are exact); the same step captured in a CUDA graph and replayed gives
the eager result bit for bit."""
import numpy as np
import pytest
import torch

import workloads as W
from dsa_cases import Shard, dsa, f64, i32, mla_close
from oracle import split as osplit

pytestmark = pytest.mark.gpu


def _decode_batch():
    wl = W.WORKLOADS[4]
    q = wl.decode_queries
    ctx = np.asarray(wl.lengths, dtype=np.int64)
    cu_new = (np.arange(len(ctx) + 1) * q).astype(np.int32)
    return wl, cu_new, (ctx - q).astype(np.int32)


def _gpu_split_decode(cu_new, pos_base, sp, rank):
    n = int(cu_new[-1])
    n_r = dsa().dsa_rr_shard_len(n, sp, rank)
    e = lambda m: torch.full((m,), -7, dtype=torch.int32, device="cuda")
    out = {"cu_shard": e(len(cu_new)), "pos": e(n_r), "bid": e(n_r), "gidx": e(n_r)}
    dsa().dsa_rr_split_decode_metadata(i32(cu_new), i32(pos_base), n, sp, rank, out["cu_shard"],
                                       out["pos"], out["bid"], out["gidx"])
    return out


@pytest.mark.parametrize("sp", [1, 2, 3, 4, 8])
def test_decode_split_matches_oracle(sp):
    _, cu_new, base = _decode_batch()
    for r in range(sp):
        g = {k: v.cpu().numpy() for k, v in _gpu_split_decode(cu_new, base, sp, r).items()}
        o = osplit.round_robin_split_decode(cu_new, base, sp, r)
        for k in ("gidx", "bid", "pos", "cu_shard"):
            assert np.array_equal(g[k], o[k]), (sp, r, k)


@pytest.mark.parametrize("seed", range(3))
def test_decode_split_random_batches(seed):
    rng = np.random.default_rng(seed)
    new = rng.integers(0, 5, int(rng.integers(1, 40)))
    cu_new = W.cu_seqlens(new)
    base = rng.integers(0, 100000, len(new)).astype(np.int32)
    sp = int(rng.integers(1, 9))
    for r in range(sp):
        g = {k: v.cpu().numpy() for k, v in _gpu_split_decode(cu_new, base, sp, r).items()}
        o = osplit.round_robin_split_decode(cu_new, base, sp, r)
        for k in ("gidx", "bid", "pos", "cu_shard"):
            assert np.array_equal(g[k], o[k]), (seed, r, k)


class DecodeShard:
    """Shard `rank` of `sp` of the decode workload: its queries are the flattened new tokens
    g = rank, rank + sp, ...; metadata comes from the decode split kernel."""

    def __init__(self, sp, rank):
        self.full = Shard(W.WORKLOADS[4], 0, integer_indexer=True)
        self.wl, cu_new, base = _decode_batch()
        self.sel = np.arange(rank, self.full.n_q, sp)
        self.meta = _gpu_split_decode(cu_new, base, sp, rank)
        sel_t = torch.as_tensor(self.sel, device="cuda")
        self.q_idx = self.full.idx.q_idx.cuda()[sel_t].contiguous()
        self.w = self.full.idx.w.cuda()[sel_t].contiguous()
        self.q = self.full.mla.q.cuda()[sel_t].contiguous()
        self.k_idx, self.c = self.full.idx.k_idx.cuda(), self.full.mla.c.cuda()
        n_q = len(self.sel)
        self.ws = torch.empty(dsa().dsa_indexer_topk_workspace_size(n_q, self.full.max_ctx,
                                                                    self.wl.topk),
                              dtype=torch.uint8, device="cuda")
        self.topk = torch.empty((n_q, self.wl.topk), dtype=torch.int32, device="cuda")
        self.o = torch.empty((n_q, self.wl.H, self.wl.dv), dtype=torch.bfloat16, device="cuda")
        self.lse = torch.empty((n_q, self.wl.H), dtype=torch.float32, device="cuda")

    def step(self):
        m, wl, f = dsa(), self.wl, self.full
        m.dsa_indexer_topk(self.q_idx, self.w, self.k_idx, f.d_cu, f.n_req, self.meta["pos"],
                           self.meta["bid"], wl.topk, f.max_ctx, self.topk, self.ws,
                           block_table=f.block_table)
        m.dsa_sparse_mla(self.q, self.c, f.d_cu, f.n_req, self.meta["bid"], self.topk, wl.scale,
                         self.o, self.lse, block_table=f.block_table)


def test_decode_shard_step_matches_oracle():
    ds = DecodeShard(4, 1)
    f = ds.full
    assert np.array_equal(ds.meta["bid"].cpu().numpy(), f.bid[ds.sel])
    assert np.array_equal(ds.meta["pos"].cpu().numpy(), f.pos[ds.sel])
    ds.step()
    view = f.oracle_view(ds.sel)
    ora_topk = f.oracle_topk(f.oracle_scores(ds.sel, view))
    assert np.array_equal(ds.topk.cpu().numpy(), ora_topk)
    ref_o, ref_lse = f.oracle_mla(ds.sel, ora_topk, view)
    mla_close(f64(ds.o), ref_o)
    assert np.allclose(ds.lse.cpu().numpy(), ref_lse, atol=1e-3, rtol=1e-4)


def test_decode_shard_step_replays_from_a_cuda_graph():
    ds = DecodeShard(8, 5)
    torch.cuda.synchronize()
    ds.step()
    torch.cuda.synchronize()
    eager_topk, eager_o = ds.topk.clone(), ds.o.clone()
    ds.topk.fill_(-9)
    ds.o.fill_(0)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):                      # warm the launch path off the capture
        ds.step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ds.step()
    ds.topk.fill_(-9)
    ds.o.fill_(0)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(ds.topk, eager_topk)
    assert torch.equal(ds.o, eager_o)
    assert dsa().dsa_read_device_errors() == 0
