"""GPU parity: tcgen05 sparse MLA vs the fp64 oracle (max-abs 2e-2 and rel-RMS 5e-3 on the
bf16 output; lse within 1e-3). Index sets come from the oracle, so the MLA is checked on its
own."""
import numpy as np
import pytest
import torch

import workloads as W
from dsa_cases import Shard, f64, i32, mla_close
from oracle import mla as omla

pytestmark = pytest.mark.gpu


def _check(sh, sel, topk_np, view=None):
    sel_t = torch.as_tensor(np.asarray(sel), device="cuda")
    o, lse = sh.run_mla(i32(topk_np), q=sh.mla.q[sel_t].cuda(), bid=i32(sh.bid[sel]))
    ref_o, ref_lse = sh.oracle_mla(sel, topk_np, view)
    ma, rr = mla_close(f64(o), ref_o)
    assert np.allclose(lse.cpu().numpy(), ref_lse, atol=1e-3, rtol=1e-4)
    return ma, rr


def test_tiny_workload_all_queries():
    sh = Shard(W.WORKLOADS[0], 1)
    sel = np.arange(sh.n_q)
    view = sh.oracle_view(sel)
    topk = sh.oracle_topk(sh.oracle_scores(sel, view))
    _check(sh, sel, topk, view)


@pytest.mark.parametrize("wid,rank", [(1, 3), (2, 6), (3, 1)])
def test_prefill_workloads_sampled(wid, rank):
    sh = Shard(W.WORKLOADS[wid], rank, integer_indexer=False)
    sel = sh.samples(48)
    view = sh.oracle_view(sel)
    topk = sh.oracle_topk(sh.oracle_scores(sel, view))
    _check(sh, sel, topk, view)


def test_paged_decode_sampled():
    sh = Shard(W.WORKLOADS[4], 0)
    sel = sh.samples(24)
    view = sh.oracle_view(sel)
    topk = sh.oracle_topk(sh.oracle_scores(sel, view))
    _check(sh, sel, topk, view)


def test_topk_covering_context_equals_dense_causal():
    sh = Shard(W.WORKLOADS[1], 3)
    sel = np.flatnonzero(sh.pos < 300)[:40]
    topk = np.full((len(sel), 2048), -1, dtype=np.int64)
    for i, t in enumerate(sel):
        topk[i, :sh.pos[t] + 1] = np.arange(sh.pos[t] + 1)
    view = sh.oracle_view(sel)
    sel_t = torch.as_tensor(sel, device="cuda")
    o, lse = sh.run_mla(i32(topk), q=sh.mla.q[sel_t].cuda(), bid=i32(sh.bid[sel]))
    ref_o, ref_lse = omla.dense_causal_mla(view["q"], view["c"], view["kv"], view["pos"],
                                           view["bid"], sh.wl.scale, sh.wl.dv)
    mla_close(f64(o), ref_o)


def test_padding_holes_and_empty_rows():
    sh = Shard(W.WORKLOADS[1], 3)
    rng = np.random.default_rng(3)
    sel = np.flatnonzero(sh.pos > 4000)[:6]
    topk = np.full((len(sel), 2048), -1, dtype=np.int64)
    for i, t in enumerate(sel):
        picks = rng.choice(sh.pos[t] + 1, 700, replace=False)
        slots = rng.choice(2048, 700, replace=False)    # valid entries scattered among -1
        topk[i, slots] = picks
    topk[-1, :] = -1                                    # a query with nothing selected
    view = sh.oracle_view(sel)
    sel_t = torch.as_tensor(sel, device="cuda")
    o, lse = sh.run_mla(i32(topk), q=sh.mla.q[sel_t].cuda(), bid=i32(sh.bid[sel]))
    ref_o, ref_lse = sh.oracle_mla(sel, topk, view)
    mla_close(f64(o), ref_o)
    assert np.all(f64(o)[-1] == 0) and np.all(np.isneginf(lse.cpu().numpy()[-1]))


@pytest.mark.parametrize("gain", [12.0, 20.0])
def test_large_logits_trigger_rescale(gain):
    """Logits scaled up 12x / 20x (std ~17 / ~29 in log2 units) make a row's running maximum
    grow past the lazy threshold after the first tile (the O-rescaling path). Outputs then reach
    |o| ~ 4-8, where one bf16 ulp of o is 2^-5, so the fixed 2e-2 absolute bound of the N(0,1)
    workloads does not apply. Bound used, elementwise: bf16 rounding of o (2^-8 |o|) plus bf16
    rounding of P (2^-8 max |v| over the selected rows), plus 1e-3; rel-RMS stays <= 5e-3."""
    sh = Shard(W.WORKLOADS[1], 3)
    sel = np.flatnonzero(sh.pos > 3000)[:4]
    idx = torch.as_tensor(sel, device=sh.mla.q.device)
    sh.mla.q = sh.mla.q.clone()
    sh.mla.q[idx] = (sh.mla.q[idx].float() * gain).to(torch.bfloat16)
    topk = np.tile(np.arange(2048), (len(sel), 1))
    view = sh.oracle_view(sel)
    o, lse = sh.run_mla(i32(topk), q=sh.mla.q[idx].cuda(), bid=i32(sh.bid[sel]))
    ref_o, ref_lse = sh.oracle_mla(sel, topk, view)
    og = f64(o)
    vmax = np.max(np.abs(view["c"][:, :sh.wl.dv]))
    bound = 2.0 ** -8 * np.abs(ref_o) + 2.0 ** -8 * vmax + 1e-3
    assert np.all(np.abs(og - ref_o) <= bound), float(np.max(np.abs(og - ref_o) / bound))
    assert np.linalg.norm(og - ref_o) / np.linalg.norm(ref_o) <= 5e-3
    assert np.allclose(lse.cpu().numpy(), ref_lse, atol=1e-3, rtol=1e-4)


@pytest.mark.parametrize("k", [1, 47, 49, 96, 4096])
def test_unusual_k(k):
    """Top-k widths that do not fill whole 48-key tiles (1, 47, 49, 96) and the largest k the
    pair kernel takes (4096, which sizes its per-query validity-mask buffer)."""
    sh = Shard(W.WORKLOADS[1], 3)
    rng = np.random.default_rng(k)
    sel = np.flatnonzero(sh.pos > 7000)[:4]
    topk = np.full((len(sel), k), -1, dtype=np.int64)
    for i, t in enumerate(sel):
        n_pick = min(k, int(sh.pos[t]) + 1)
        topk[i, :n_pick] = np.sort(rng.choice(int(sh.pos[t]) + 1, n_pick, replace=False))
    _check(sh, sel, topk)


@pytest.mark.parametrize("balanced", [False, True])
def test_out_of_range_entries_are_skipped_and_flagged(balanced):
    """Entries past the query's position (balanced call, which is given the positions) or past
    its request's end (both calls, contiguous KV) are not attended: they are skipped like -1
    padding and DEVERR_BAD_INDEX is set. The output equals the oracle over the remaining
    entries."""
    from dsa_cases import dsa
    sh = Shard(W.WORKLOADS[1], 3)
    rng = np.random.default_rng(11)
    # queries of request 1 (800 tokens, rows 8000..8799) and request 3 (3000 tokens)
    sel = np.concatenate([np.flatnonzero(sh.bid == 1)[20:23], np.flatnonzero(sh.bid == 3)[100:103]])
    k = 256
    topk = np.full((len(sel), k), -1, dtype=np.int64)
    keep = np.full((len(sel), k), -1, dtype=np.int64)
    for i, t in enumerate(sel):
        p = int(sh.pos[t])
        L = int(sh.cu[sh.bid[t] + 1] - sh.cu[sh.bid[t]])
        good = rng.choice(p + 1, min(150, p + 1), replace=False)
        past_req = L + rng.integers(0, 50, 3)                 # beyond the request: always invalid
        past_pos = p + 1 + rng.integers(0, L - p - 1, 3) if L - p - 1 > 0 else np.zeros(0, int)
        ent = np.concatenate([good, past_req, past_pos])
        slots = rng.choice(k, len(ent), replace=False)
        topk[i, slots] = ent
        valid = (ent <= p) if balanced else (ent < L)
        keep[i, slots[valid]] = ent[valid]
    m = dsa()
    q = sh.mla.q[torch.as_tensor(sel, device=sh.mla.q.device)].cuda()
    o = torch.full((len(sel), 128, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((len(sel), 128), float("nan"), device="cuda")
    m.dsa_read_device_errors()
    bid, pos = i32(sh.bid[sel]), i32(sh.pos[sel])
    if balanced:
        ws = torch.empty(m.dsa_sparse_mla_workspace_size(len(sel)), dtype=torch.uint8, device="cuda")
        m.dsa_sparse_mla_balanced(q, sh.mla.c.cuda(), sh.d_cu, sh.n_req, bid, pos, i32(topk),
                                  sh.wl.scale, o, ws, lse=lse)
    else:
        m.dsa_sparse_mla(q, sh.mla.c.cuda(), sh.d_cu, sh.n_req, bid, i32(topk), sh.wl.scale, o, lse)
    assert m.dsa_read_device_errors() & m.DEVERR_BAD_INDEX
    # the oracle over the entries that stay (the plain call keeps entries past pos but inside
    # the request; they are real keys of the request, so the oracle reads them too)
    cu = sh.cu.astype(np.int64)
    c64 = f64(sh.mla.c)
    from oracle.kv import ContiguousKV
    ref_o, ref_lse = omla.sparse_mla(f64(q), c64, ContiguousKV(cu), sh.bid[sel], keep,
                                     sh.wl.scale, sh.wl.dv)
    mla_close(f64(o), ref_o)
    assert np.allclose(lse.cpu().numpy(), ref_lse, atol=1e-3, rtol=1e-4)
