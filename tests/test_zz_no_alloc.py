"""The allocation-free indexer + top-k entry point (for callers that cannot allocate device
memory) gives the same index sets as the entry point that takes a caller workspace.

Kept in its own file, collected last, so that a failure here does not hide other results."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from dsa_cases import Shard

pytestmark = pytest.mark.gpu


def _noalloc_via_c_abi(sh):
    """Call the C entry point directly through ctypes (no workspace argument exists)."""
    from deepseek_v3_sparse_round_gb300 import _native
    lib = _native.load()
    topk = torch.full((sh.n_q, sh.wl.topk), -9, dtype=torch.int32, device="cuda")
    q_idx, w, k_idx = sh.idx.q_idx.cuda(), sh.idx.w.cuda(), sh.idx.k_idx.cuda()
    bt = sh.block_table
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    rc = lib.dsa_indexer_topk_noalloc(
        p(q_idx), p(w), p(k_idx), k_idx.shape[0], p(sh.d_cu), sh.n_req, p(sh.d_pos), p(sh.d_bid),
        sh.n_q, sh.wl.Hi, sh.wl.Di, sh.wl.topk, sh.max_ctx, p(bt),
        bt.shape[1] if bt is not None else 0, 64, p(topk),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, lib.dsa_last_error_string()
    torch.cuda.synchronize()
    return topk


def test_two_calls_in_a_row_match_the_workspace_entry_point():
    # bf16 N(0,1) indexer inputs; the two paths run the same kernels, so the index sets agree
    # exactly (the tolerance for index work is bit-exactness).
    first = Shard(W.WORKLOADS[1], 3)
    second = Shard(W.WORKLOADS[0], 1)
    for sh in (first, second):
        got = _noalloc_via_c_abi(sh)
        ref = sh.run_indexer_topk()
        torch.cuda.synchronize()
        assert torch.equal(got, ref)
    again = _noalloc_via_c_abi(first)        # the array keeps the previous call's contents
    assert torch.equal(again, first.run_indexer_topk())


def test_oversized_request_is_rejected():
    from deepseek_v3_sparse_round_gb300 import _native
    lib = _native.load()
    fake = ctypes.c_void_p(4096)
    rc = lib.dsa_indexer_topk_noalloc(fake, fake, fake, 10, fake, 1, fake, fake, 1 << 20, 64, 128,
                                      2048, 65536, None, 0, 64, fake, None)
    assert rc == -3 and b"static" in lib.dsa_last_error_string()
