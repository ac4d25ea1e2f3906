"""The C-ABI library builds for sm_103a, loads, and exports every function include/dsa_rr.h
declares; host-side helpers and argument validation work without a GPU."""
import ctypes
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def lib():
    from deepseek_v3_sparse_round_gb300 import build as b
    from deepseek_v3_sparse_round_gb300 import _native
    b.build()
    return _native.load()


def _declared():
    with open(os.path.join(ROOT, "include", "dsa_rr.h"), encoding="utf-8") as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    from deepseek_v3_sparse_round_gb300._native import SIGNATURES
    assert sorted(SIGNATURES) == names


def test_library_is_sm103a_build():
    from deepseek_v3_sparse_round_gb300 import build as b
    assert "arch=compute_103a,code=sm_103a" in " ".join(b.ARCH)


def test_host_helpers(lib):
    import deepseek_v3_sparse_round_gb300 as dsa
    assert dsa.dsa_version() == 1
    assert dsa.dsa_rr_shard_len(11805, 8, 3) == 1476
    assert dsa.dsa_rr_shard_len(3, 8, 5) == 0
    assert dsa.dsa_rr_shard_len(0, 4, 0) == 0
    assert dsa.dsa_rr_shard_len(10, 0, 0) == -1 and dsa.dsa_rr_shard_len(10, 4, 4) == -1
    assert sum(dsa.dsa_rr_shard_len(71014, 4, r) for r in range(4)) == 71014
    assert dsa.dsa_score_row_stride(8001) == 8004
    ws = dsa.dsa_indexer_topk_workspace_size(1476, 8000, 2048)
    assert ws >= 1476 * 8000 * 4 and ws % 256 == 0


def test_invalid_arguments_rejected_before_any_launch(lib):
    null = ctypes.c_void_p(0)
    # sp = 0, rank >= sp, n_req = 0
    assert lib.dsa_rr_split_metadata(null, 1, 10, 0, 0, null, null, null, null, null, null, 0, null) == -1
    assert lib.dsa_rr_split_metadata(null, 1, 10, 4, 4, null, null, null, null, null, null, 0, null) == -1
    assert b"sp" in lib.dsa_last_error_string()
    assert lib.dsa_rr_rerange(null, null, 10, 4, 1, 16, null) == -1          # stride < ceil(N/sp)
    assert lib.dsa_rr_rerange(null, null, 0, 4, 0, 16, null) == 0            # empty is a no-op
    # unsupported shapes and missing workspace
    fake = ctypes.c_void_p(4096)
    assert lib.dsa_sparse_mla(fake, fake, 10, fake, 1, fake, fake, 4, 64, 576, 512, 2048, 0.1,
                              null, 0, 0, fake, null, null) == -2
    assert lib.dsa_sparse_mla(fake, fake, 10, fake, 1, fake, fake, 4, 128, 576, 512, 8192, 0.1,
                              null, 0, 0, fake, null, null) == -2
    assert lib.dsa_indexer_topk(fake, fake, fake, 10, fake, 1, fake, fake, 4, 64, 128, 2048, 10,
                                null, 0, 0, fake, null, 0, null) == -3
    assert lib.dsa_topk_select(fake, 3, fake, 4, 8, 10, fake, null) == -1    # stride < max_ctx
    assert lib.dsa_indexer_scores(fake, fake, fake, 10, fake, 1, fake, fake, 4, 32, 128, 10, null,
                                  0, 0, fake, 12, fake, 1 << 20, null) == -2


def test_rerange_paged_arguments_rejected(lib):
    null = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(4096)
    f = lib.dsa_rr_rerange_paged
    assert f(fake, fake, 64, 10, 0, 0, 16, fake, 1, fake, 1, 64, null) == -1     # sp = 0
    assert f(fake, fake, 64, 10, 4, 1, 16, fake, 1, fake, 1, 64, null) == -1     # stride < ceil(N/sp)
    assert f(fake, fake, 64, 10, 4, 0, 16, fake, 1, fake, 1, 0, null) == -1      # page_size 0
    assert f(fake, fake, 64, 10, 4, 0, 16, fake, 0, fake, 1, 64, null) == -1     # n_req 0
    assert f(null, fake, 64, 10, 4, 0, 16, fake, 1, fake, 1, 64, null) == -1     # null gathered
    assert f(null, null, 0, 0, 4, 0, 16, null, 1, null, 1, 64, null) == 0        # empty no-op


def test_split_decode_needs_pos_base(lib):
    null = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(4096)
    f = lib.dsa_rr_split_decode_metadata
    assert f(fake, null, 1, 10, 4, 0, fake, fake, fake, null, null, null, 0, null) == -1
    assert b"pos_base" in lib.dsa_last_error_string()
    assert f(fake, fake, 1, 10, 0, 0, fake, fake, fake, null, null, null, 0, null) == -1   # sp = 0


def test_sparse_mla_balanced_arguments_rejected(lib):
    null = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(4096)
    f = lib.dsa_sparse_mla_balanced
    args = lambda pos, ws, ws_bytes: (fake, fake, 10, fake, 1, fake, pos, fake, 4, 128, 576, 512,
                                      2048, 0.1, null, 0, 0, fake, null, ws, ws_bytes, null)
    assert f(*args(null, fake, 16)) == -1                              # pos is required
    assert b"pos" in lib.dsa_last_error_string()
    assert f(*args(fake, fake, 8)) == -3                               # 4 queries need 16 bytes
    assert f(*args(fake, null, 16)) == -3                              # no workspace
    assert f(*args(fake, ctypes.c_void_p(4100), 16)) == -1             # not 16-byte aligned
    assert lib.dsa_sparse_mla_workspace_size(1476) == 1476 * 4
    assert lib.dsa_sparse_mla_workspace_size(0) == 0


def test_sparse_mla_shapes_rejected_before_any_launch(lib):
    """Widths and shapes the MLA kernels are not built for, and misaligned q / o, come back as
    return codes from host checks (no device memory is touched)."""
    null, fake = ctypes.c_void_p(0), ctypes.c_void_p(4096)
    f = lib.dsa_sparse_mla

    def call(k=2048, H=128, dqk=576, dv=512, q=fake, o=fake, page_size=64, table=null):
        return f(q, fake, 1000, fake, 1, fake, fake, 4, H, dqk, dv, k, 0.05, table, 1, page_size,
                 o, null, null)

    assert call(k=4097) == -2                                          # beyond the 4096-wide mask
    assert call(H=64) == -2 and call(dqk=512) == -2 and call(dv=256) == -2
    assert call(k=0) == -1
    assert call(q=ctypes.c_void_p(4100)) == -1                         # q not 16-byte aligned
    assert call(o=ctypes.c_void_p(4104)) == -1                         # o not 16-byte aligned
    assert call(table=fake, page_size=32) == -2                        # pages of 64 tokens only
    assert f(null, fake, 1000, fake, 1, fake, fake, 4, 128, 576, 512, 2048, 0.05, null, 1, 64,
             fake, null, null) == -1                                   # null q
