"""Shared staging for the GPU parity tests: inputs from `workloads`, the CUDA path through the
Python binding of the C ABI, and the fp64 oracle on the CPU. The two sides share only inputs."""
from __future__ import annotations

import numpy as np
import torch

import workloads as W
from oracle import indexer as oidx
from oracle import mla as omla
from oracle import split as osplit
from oracle import topk as otopk
from oracle.kv import ContiguousKV, PagedKV


def dsa():
    import deepseek_v3_sparse_round_gb300 as m
    return m


def i32(a, device="cuda"):
    return torch.as_tensor(np.ascontiguousarray(np.asarray(a, dtype=np.int32)), device=device)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


# ----------------------------------------------------------------------------- split / rerange
def gpu_split(cu_np, sp, rank, src=None):
    n = int(cu_np[-1])
    n_r = dsa().dsa_rr_shard_len(n, sp, rank)
    cu = i32(cu_np)
    out = {k: torch.full((n_r,), -7, dtype=torch.int32, device="cuda") for k in ("pos", "bid", "gidx")}
    cu_shard = torch.full((len(cu_np),), -7, dtype=torch.int32, device="cuda")
    dst = None
    if src is not None:
        dst = torch.empty((n_r,) + tuple(src.shape[1:]), dtype=src.dtype, device="cuda")
    dsa().dsa_rr_split_metadata(cu, n, sp, rank, cu_shard, out["pos"], out["bid"], out["gidx"],
                                src_rows=src, dst_rows=dst)
    res = {k: v.cpu().numpy() for k, v in out.items()}
    res["cu_shard"] = cu_shard.cpu().numpy()
    res["rows"] = dst
    return res


def gpu_gather_and_rerange(logical: torch.Tensor, cu_np, sp, padded: bool):
    """Each rank's rows by the split kernel, concatenated rank by rank (the all-gather layout),
    then put back in logical order by the rerange kernel."""
    n = logical.shape[0]
    shards = [gpu_split(cu_np, sp, r, src=logical)["rows"] for r in range(sp)]
    stride = (-(-n // sp)) if padded else 0
    if padded:
        blocks = []
        for s in shards:
            pad = torch.zeros((stride - s.shape[0],) + tuple(s.shape[1:]), dtype=s.dtype, device="cuda")
            blocks.append(torch.cat([s, pad]))
        gathered = torch.cat(blocks)
    else:
        gathered = torch.cat(shards)
    out = torch.empty_like(logical)
    dsa().dsa_rr_rerange(gathered, out, n, sp, stride)
    return gathered, out


# ----------------------------------------------------------------------------- shard staging
class Shard:
    """One shard of a workload: metadata, inputs, and the CUDA path's outputs."""

    def __init__(self, wl: W.Workload, rank: int, integer_indexer=None, gen_device="cuda"):
        self.wl, self.rank = wl, rank
        if wl.decode_queries:
            self.ctx = np.asarray(wl.lengths, dtype=np.int64)
            self.bid, self.pos = W.decode_queries(wl.lengths, wl.decode_queries)
            self.table, n_pages = W.random_block_table(wl.lengths, wl.page_size,
                                                       W.seed_of(wl, "block_table"))
            self.n_rows = n_pages * wl.page_size
            self.cu = np.zeros(len(wl.lengths) + 1, dtype=np.int32)   # unused when paged
            self.kv = PagedKV(self.table, wl.page_size)
            self.max_ctx = int(self.ctx.max())
            self.block_table = i32(self.table)
        else:
            self.cu = W.cu_seqlens(wl.lengths)
            meta = osplit.round_robin_split(self.cu, wl.sp, rank)
            self.bid, self.pos = meta["bid"].astype(np.int32), meta["pos"].astype(np.int32)
            self.n_rows = int(self.cu[-1])
            self.kv = ContiguousKV(self.cu)
            self.max_ctx = int(max(wl.lengths))
            self.block_table = None
        self.n_q = len(self.pos)
        self.n_req = len(wl.lengths)
        self.idx = W.indexer_inputs(wl, self.n_q, self.n_rows, rank, integer=integer_indexer,
                                    device=gen_device)
        self.mla = W.mla_inputs(wl, self.n_q, self.n_rows, rank, device=gen_device)
        self.d_cu, self.d_pos, self.d_bid = i32(self.cu), i32(self.pos), i32(self.bid)

    # --- CUDA path ---
    def run_indexer(self):
        m = dsa()
        stride = m.dsa_score_row_stride(self.max_ctx)
        self.scores = torch.full((self.n_q, stride), float("nan"), device="cuda")
        ws = torch.empty(m.dsa_indexer_topk_workspace_size(self.n_q, self.max_ctx, self.wl.topk),
                         dtype=torch.uint8, device="cuda")
        m.dsa_indexer_scores(self.idx.q_idx.cuda(), self.idx.w.cuda(), self.idx.k_idx.cuda(),
                             self.d_cu, self.n_req, self.d_pos, self.d_bid, self.max_ctx,
                             self.scores, ws, block_table=self.block_table)
        self.topk = torch.full((self.n_q, self.wl.topk), -9, dtype=torch.int32, device="cuda")
        m.dsa_topk_select(self.scores, self.d_pos, self.wl.topk, self.max_ctx, self.topk)
        return self.scores, self.topk

    def run_indexer_topk(self, k=None):
        m = dsa()
        k = self.wl.topk if k is None else k
        ws = torch.empty(m.dsa_indexer_topk_workspace_size(self.n_q, self.max_ctx, k),
                         dtype=torch.uint8, device="cuda")
        topk = torch.full((self.n_q, k), -9, dtype=torch.int32, device="cuda")
        m.dsa_indexer_topk(self.idx.q_idx.cuda(), self.idx.w.cuda(), self.idx.k_idx.cuda(), self.d_cu,
                           self.n_req, self.d_pos, self.d_bid, k, self.max_ctx, topk, ws,
                           block_table=self.block_table)
        return topk

    def run_mla(self, topk: torch.Tensor, q=None, bid=None):
        m = dsa()
        q = self.mla.q.cuda() if q is None else q
        bid = self.d_bid if bid is None else bid
        o = torch.full((q.shape[0], self.wl.H, self.wl.dv), float("nan"), dtype=torch.bfloat16,
                       device="cuda")
        lse = torch.full((q.shape[0], self.wl.H), float("nan"), device="cuda")
        m.dsa_sparse_mla(q, self.mla.c.cuda(), self.d_cu, self.n_req, bid, topk, self.wl.scale, o, lse,
                         block_table=self.block_table)
        return o, lse

    # --- oracle on a subset of queries ---
    def oracle_view(self, sel):
        """fp64 inputs for queries `sel`: the KV rows of their requests (positions 0..max pos,
        located by the oracle's own row map) packed per request, with re-numbered requests."""
        sel = np.asarray(sel, dtype=np.int64)
        reqs = sorted(set(int(b) for b in self.bid[sel]))
        need = {b: int(self.pos[sel][self.bid[sel] == b].max()) + 1 for b in reqs}
        rows = np.concatenate([self.kv.rows(b, np.arange(need[b])) for b in reqs])
        cu2 = np.concatenate([[0], np.cumsum([need[b] for b in reqs])]).astype(np.int64)
        remap = {b: i for i, b in enumerate(reqs)}
        r = torch.as_tensor(rows, device=self.idx.k_idx.device)
        view = {
            "q_idx": f64(self.idx.q_idx[torch.as_tensor(sel, device=self.idx.q_idx.device)]),
            "w": f64(self.idx.w[torch.as_tensor(sel, device=self.idx.w.device)]),
            "k_idx": f64(self.idx.k_idx[r]),
            "q": f64(self.mla.q[torch.as_tensor(sel, device=self.mla.q.device)]),
            "c": f64(self.mla.c[r.to(self.mla.c.device)]),
            "kv": ContiguousKV(cu2),
            "pos": self.pos[sel],
            "bid": np.asarray([remap[int(b)] for b in self.bid[sel]], dtype=np.int64),
            "row_ids": rows,                             # the view's rows in the full tensors
        }
        return view

    def oracle_scores(self, sel, view=None):
        v = self.oracle_view(sel) if view is None else view
        return oidx.indexer_scores(v["q_idx"], v["w"], v["k_idx"], v["kv"], v["pos"], v["bid"])

    def oracle_topk(self, rows):
        return otopk.topk_rows(rows, self.wl.topk)

    def oracle_mla(self, sel, topk_np, view=None):
        v = self.oracle_view(sel) if view is None else view
        return omla.sparse_mla(v["q"], v["c"], v["kv"], v["bid"], topk_np, self.wl.scale,
                               self.wl.dv)

    def samples(self, n_sample=64, seed=0):
        """First and last query of every request plus random others."""
        must = []
        for b in range(self.n_req):
            ids = np.flatnonzero(self.bid == b)
            if len(ids):
                must += [ids[0], ids[-1]]
        return W.sample_queries(self.n_q, np.asarray(must, dtype=np.int64), n_sample, seed)


def score_error_bound(view, t_local, s_count, Di, Hi):
    """Elementwise bound on |fp32 tensor-core score - exact score| for query t_local of an
    oracle view: each bf16 product is exact in fp32, and the fp32 sums over Di and then Hi
    terms each lose at most (terms) * 2^-24 of the sum of magnitudes; 2^-22 (Di + Hi) leaves a
    4x margin."""
    q = np.abs(view["q_idx"][t_local])                  # [Hi, Di]
    w = np.abs(view["w"][t_local])                      # [Hi]
    keys = np.abs(view["k_idx"][view["kv"].rows(int(view["bid"][t_local]), np.arange(s_count))])
    mag = w @ (q @ keys.T)                              # [s_count]
    return 2.0 ** -22 * (Di + Hi) * mag + 1e-30


def check_topk_near_ties(gpu_idx, ora_idx, exact_scores, k, rel=1e-3):
    """Index sets may differ only between entries whose exact scores sit within tau of the
    oracle's k-th score, tau = rel * max |score| of the row."""
    g = set(int(x) for x in gpu_idx if x >= 0)
    o = set(int(x) for x in ora_idx if x >= 0)
    assert len(g) == len(o), (len(g), len(o))
    if g == o:
        return 0
    kth = np.sort(exact_scores)[::-1][min(k, len(exact_scores)) - 1]
    tau = rel * np.max(np.abs(exact_scores))
    for s in g ^ o:
        assert abs(exact_scores[s] - kth) <= tau, (s, exact_scores[s], kth, tau)
    return len(g ^ o) // 2


def mla_close(o_gpu: np.ndarray, o_ref: np.ndarray, max_abs=2e-2, rel_rms=5e-3):
    d = o_gpu - o_ref
    ma = float(np.max(np.abs(d))) if d.size else 0.0
    rr = float(np.linalg.norm(d) / max(np.linalg.norm(o_ref), 1e-30)) if d.size else 0.0
    assert ma <= max_abs and rr <= rel_rms, f"max-abs {ma:.3e} (<= {max_abs}), rel-RMS {rr:.3e} (<= {rel_rms})"
    return ma, rr
