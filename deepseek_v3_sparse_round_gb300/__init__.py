"""Round-robin sequence-shard DSA prefill attention for GB300 (sm_103a).

Python binding of the C ABI in include/dsa_rr.h. Every function here only marshals arguments
(torch tensors -> device pointers, the current CUDA stream) and calls the native library of the
same name; all computation runs in the library's CUDA kernels. If libdsa_rr.so is missing the
calls raise: there is no CPU or PyTorch fallback.
"""
from __future__ import annotations

import ctypes
import math

import torch

from . import _native

__all__ = [
    "DsaError", "dsa_version", "dsa_rr_shard_len", "dsa_rr_split_metadata", "dsa_rr_rerange",
    "dsa_rr_rerange_paged", "dsa_rr_split_decode_metadata", "dsa_rr_rerange_multi",
    "dsa_indexer_topk_workspace_size", "dsa_score_row_stride", "dsa_indexer_scores",
    "dsa_topk_select", "dsa_indexer_topk", "dsa_indexer_topk_noalloc", "dsa_sparse_mla",
    "dsa_sparse_mla_workspace_size", "dsa_sparse_mla_balanced", "dsa_read_device_errors",
    "dsa_rr_cache_local_paged", "dsa_selftest_bounded_wait", "dsa_probe_row_gather",
    "dsa_quantize_fp8_rows", "dsa_quantize_fp8_latent", "dsa_dequantize_fp8_latent",
    "FP8_LATENT_ROW_BYTES",
    "dsa_indexer_scores_fp8", "dsa_indexer_topk_fp8",
    "DEVERR_TIMEOUT", "DEVERR_BAD_INDEX", "DEVERR_BAD_LENGTH",
]

DEVERR_TIMEOUT = 0x80000000
DEVERR_BAD_INDEX = 0x40000000
DEVERR_BAD_LENGTH = 0x20000000


class DsaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"dsa error {code}: {msg}")
        self.code = code


def _lib():
    return _native.load()


def _check(rc: int):
    if rc != 0:
        raise DsaError(rc, _lib().dsa_last_error_string().decode(errors="replace"))


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if t.numel() > 0 and not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _dev(t, dtype=None, name="tensor"):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _shape(t, want, name):
    """Raise ValueError unless t's shape matches `want` (None entries match any size). The C ABI
    takes bare pointers and cannot check sizes, so the binding does, before any launch."""
    if t is None:
        return
    got = tuple(t.shape)
    if len(got) != len(want) or any(w is not None and g != w for g, w in zip(got, want)):
        raise ValueError(f"{name} has shape {got}, expected {tuple('*' if w is None else w for w in want)}")


def _row_bytes(t):
    return math.prod(t.shape[1:]) * t.element_size()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def dsa_version() -> int:
    return _lib().dsa_version()


def dsa_rr_shard_len(n_tokens: int, sp: int, rank: int) -> int:
    return int(_lib().dsa_rr_shard_len(n_tokens, sp, rank))


def dsa_score_row_stride(max_ctx: int) -> int:
    return int(_lib().dsa_score_row_stride(max_ctx))


def dsa_indexer_topk_workspace_size(n_q: int, max_ctx: int, k: int) -> int:
    return int(_lib().dsa_indexer_topk_workspace_size(n_q, max_ctx, k))


def dsa_read_device_errors() -> int:
    flags = ctypes.c_uint32(0)
    _check(_lib().dsa_read_device_errors(ctypes.byref(flags)))
    return int(flags.value)


def dsa_selftest_bounded_wait(limit_cycles: int, stream=None):
    """One kernel waits, with the library's bounded wait, on a phase nothing completes; after
    limit_cycles the wait gives up and sets DEVERR_TIMEOUT | 0xEE (read it with
    dsa_read_device_errors)."""
    _check(_lib().dsa_selftest_bounded_wait(int(limit_cycles), _stream(stream)))


def dsa_probe_row_gather(c, rows, n_ctas, n_tiles, mode, issuers, cycles, stream=None):
    """Row-gather rate probe: c bf16 [n_rows, 576]; rows int32 [n_ctas * n_tiles * 48];
    mode 0 = cp.async (three warps per ring slot), 1 = TMA tile::gather4 by `issuers` lanes,
    2 = columns 0..511 by cp.async and 512..575 by tile::gather4, 3 = DSMEM push between the
    CTAs of pairs (192 KB per round, n_tiles rounds), 4 = as 0 through registers, 5 = columns
    0..319 through registers and 320..575 by cp.async, 6 = as 4 with all rows in flight,
    7 = TMA tiled boxes of the 48 consecutive rows from each tile's first listed row; cycles int64 [n_ctas] receives each CTA's loop time in SM clock cycles."""
    _dev(c, torch.bfloat16, "c")
    _dev(rows, torch.int32, "rows")
    _dev(cycles, torch.int64, "cycles")
    if c.dim() != 2 or c.shape[1] != 576:
        raise ValueError(f"c must be [n_rows, 576], got {tuple(c.shape)}")
    _shape(rows, (int(n_ctas) * int(n_tiles) * 48,), "rows")
    _shape(cycles, (int(n_ctas),), "cycles")
    _check(_lib().dsa_probe_row_gather(_ptr(c), c.shape[0], _ptr(rows), int(n_ctas), int(n_tiles),
                                       int(mode), int(issuers), _ptr(cycles), _stream(stream)))


def dsa_rr_split_metadata(cu, n_tokens, sp, rank, cu_shard, pos, bid, gidx=None,
                          src_rows=None, dst_rows=None, stream=None):
    """cu int32 [B+1] -> cu_shard [B+1], pos/bid/gidx [n_r]; optional dst_rows = src_rows[g_t]."""
    for name, t in (("cu", cu), ("cu_shard", cu_shard), ("pos", pos), ("bid", bid), ("gidx", gidx)):
        _dev(t, torch.int32, name)
    n_r = max(0, int(_lib().dsa_rr_shard_len(n_tokens, sp, rank)))
    _shape(cu_shard, (cu.numel(),), "cu_shard")
    for name, t in (("pos", pos), ("bid", bid), ("gidx", gidx)):
        _shape(t, (n_r,), name)
    row_bytes = 0
    if src_rows is not None:
        _dev(src_rows, None, "src_rows")
        _dev(dst_rows, src_rows.dtype, "dst_rows")
        if src_rows.shape[0] < n_tokens or dst_rows.shape[0] < n_r or \
                tuple(dst_rows.shape[1:]) != tuple(src_rows.shape[1:]):
            raise ValueError("src_rows needs n_tokens rows and dst_rows n_r rows of the same width")
        row_bytes = _row_bytes(src_rows)
    _check(_lib().dsa_rr_split_metadata(_ptr(cu), cu.numel() - 1, n_tokens, sp, rank,
                                        _ptr(cu_shard), _ptr(pos), _ptr(bid), _ptr(gidx),
                                        _ptr(src_rows), _ptr(dst_rows), row_bytes,
                                        _stream(stream)))


def dsa_rr_split_decode_metadata(cu_new, pos_base, n_tokens, sp, rank, cu_shard, pos, bid,
                                 gidx=None, src_rows=None, dst_rows=None, stream=None):
    """As dsa_rr_split_metadata over a decode step's new tokens; pos = pos_base[b] + index."""
    for name, t in (("cu_new", cu_new), ("pos_base", pos_base), ("cu_shard", cu_shard),
                    ("pos", pos), ("bid", bid), ("gidx", gidx)):
        _dev(t, torch.int32, name)
    n_r = max(0, int(_lib().dsa_rr_shard_len(n_tokens, sp, rank)))
    _shape(cu_shard, (cu_new.numel(),), "cu_shard")
    _shape(pos_base, (cu_new.numel() - 1,), "pos_base")
    for name, t in (("pos", pos), ("bid", bid), ("gidx", gidx)):
        _shape(t, (n_r,), name)
    row_bytes = 0
    if src_rows is not None:
        _dev(src_rows, None, "src_rows")
        _dev(dst_rows, src_rows.dtype, "dst_rows")
        if src_rows.shape[0] < n_tokens or dst_rows.shape[0] < n_r or \
                tuple(dst_rows.shape[1:]) != tuple(src_rows.shape[1:]):
            raise ValueError("src_rows needs n_tokens rows and dst_rows n_r rows of the same width")
        row_bytes = _row_bytes(src_rows)
    _check(_lib().dsa_rr_split_decode_metadata(
        _ptr(cu_new), _ptr(pos_base), cu_new.numel() - 1, n_tokens, sp, rank, _ptr(cu_shard),
        _ptr(pos), _ptr(bid), _ptr(gidx), _ptr(src_rows), _ptr(dst_rows), row_bytes,
        _stream(stream)))


def dsa_rr_rerange(gathered, out, n_tokens, sp, rank_stride_rows=0, stream=None):
    """out[g] = gathered[off[g % sp] + g // sp] (padded blocks if rank_stride_rows > 0)."""
    _dev(gathered, None, "gathered")
    _dev(out, gathered.dtype, "out")
    need = sp * rank_stride_rows if rank_stride_rows > 0 else n_tokens
    if out.shape[0] < n_tokens or gathered.shape[0] < need or \
            tuple(out.shape[1:]) != tuple(gathered.shape[1:]):
        raise ValueError(f"rerange needs gathered with >= {need} rows and out with >= {n_tokens} "
                         "rows of the same width")
    row_bytes = _row_bytes(out)
    _check(_lib().dsa_rr_rerange(_ptr(gathered), _ptr(out), n_tokens, sp, rank_stride_rows,
                                 row_bytes, _stream(stream)))


def dsa_rr_rerange_multi(gathered, out, n_tokens, sp, rank_stride_rows=0, stream=None):
    """dsa_rr_rerange of every (gathered[q], out[q]) pair in one launch (same row map)."""
    if len(gathered) != len(out) or not gathered:
        raise ValueError("gathered and out must be non-empty lists of the same length")
    need = sp * rank_stride_rows if rank_stride_rows > 0 else n_tokens
    for g, o in zip(gathered, out):
        _dev(g, None, "gathered"); _dev(o, g.dtype, "out")
        if o.shape[0] < n_tokens or g.shape[0] < need or tuple(o.shape[1:]) != tuple(g.shape[1:]):
            raise ValueError(f"rerange needs gathered with >= {need} rows and out with >= "
                             f"{n_tokens} rows of the same width")
    n = len(gathered)
    srcs = (ctypes.c_void_p * n)(*[g.data_ptr() for g in gathered])
    dsts = (ctypes.c_void_p * n)(*[o.data_ptr() for o in out])
    rb = (ctypes.c_int64 * n)(*[_row_bytes(o) for o in out])
    _check(_lib().dsa_rr_rerange_multi(srcs, dsts, rb, n, n_tokens, sp, rank_stride_rows,
                                       _stream(stream)))


def dsa_rr_rerange_paged(gathered, pool, n_tokens, sp, cu, block_table, rank_stride_rows=0,
                         page_size=64, stream=None):
    """pool[page row of (b, s)] = gathered[off[g % sp] + g // sp] for every logical token g
    (request b, position s = g - cu[b]); n_tokens = cu[-1], passed from the host."""
    _dev(gathered, None, "gathered")
    _dev(pool, gathered.dtype, "pool")
    _dev(cu, torch.int32, "cu"); _dev(block_table, torch.int32, "block_table")
    need = sp * rank_stride_rows if rank_stride_rows > 0 else n_tokens
    if gathered.shape[0] < need or tuple(pool.shape[1:]) != tuple(gathered.shape[1:]):
        raise ValueError(f"gathered needs >= {need} rows of the pool's width")
    _shape(block_table, (cu.numel() - 1, None), "block_table")
    row_bytes = _row_bytes(pool)
    _check(_lib().dsa_rr_rerange_paged(
        _ptr(gathered), _ptr(pool), pool.shape[0], n_tokens, sp, rank_stride_rows, row_bytes,
        _ptr(cu), cu.numel() - 1, _ptr(block_table), block_table.shape[1], page_size,
        _stream(stream)))


def dsa_rr_cache_local_paged(local_rows, pool, n_tokens, sp, rank, cu, block_table, page_size=64,
                             stream=None):
    """This rank's own tokens only: pool[page row of (b, j)] = local_rows[t], j = t - cu_shard[b]
    (the token's index among request b's tokens on this rank); n_tokens = cu[-1]."""
    _dev(local_rows, None, "local_rows")
    _dev(pool, local_rows.dtype, "pool")
    _dev(cu, torch.int32, "cu"); _dev(block_table, torch.int32, "block_table")
    n_r = max(0, int(_lib().dsa_rr_shard_len(n_tokens, sp, rank)))
    if local_rows.shape[0] < n_r or tuple(pool.shape[1:]) != tuple(local_rows.shape[1:]):
        raise ValueError(f"local_rows needs >= {n_r} rows of the pool's width")
    _shape(block_table, (cu.numel() - 1, None), "block_table")
    _check(_lib().dsa_rr_cache_local_paged(
        _ptr(local_rows), _ptr(pool), pool.shape[0], n_tokens, sp, rank, _row_bytes(pool),
        _ptr(cu), cu.numel() - 1, _ptr(block_table), block_table.shape[1], page_size,
        _stream(stream)))


def dsa_indexer_scores(q_idx, w, k_idx, cu, n_req, pos, bid, max_ctx, scores, workspace,
                       block_table=None, page_size=64, stream=None):
    """scores[t, s] = sum_h w[t,h] relu(q_idx[t,h] . k_idx[row(b_t, s)]) for s <= pos_t."""
    _dev(q_idx, torch.bfloat16, "q_idx"); _dev(k_idx, torch.bfloat16, "k_idx")
    _dev(w, torch.float32, "w"); _dev(scores, torch.float32, "scores")
    _dev(pos, torch.int32, "pos"); _dev(bid, torch.int32, "bid"); _dev(cu, torch.int32, "cu")
    _dev(block_table, torch.int32, "block_table")
    n_q, Hi, Di = q_idx.shape
    _indexer_shapes(q_idx, w, pos, bid, block_table, n_req)
    _shape(scores, (n_q, None), "scores")
    max_pages = block_table.shape[1] if block_table is not None else 0
    _check(_lib().dsa_indexer_scores(
        _ptr(q_idx), _ptr(w), _ptr(k_idx), k_idx.shape[0], _ptr(cu), n_req, _ptr(pos), _ptr(bid),
        n_q, Hi, Di, max_ctx, _ptr(block_table), max_pages, page_size, _ptr(scores),
        scores.shape[1], _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def _indexer_shapes(q_idx, w, pos, bid, block_table, n_req):
    n_q, Hi, _ = q_idx.shape
    _shape(w, (n_q, Hi), "w")
    _shape(pos, (n_q,), "pos")
    _shape(bid, (n_q,), "bid")
    _shape(block_table, (n_req, None), "block_table")


def dsa_topk_select(scores, pos, k, max_ctx, topk, stream=None):
    _dev(scores, torch.float32, "scores"); _dev(pos, torch.int32, "pos")
    _dev(topk, torch.int32, "topk")
    _shape(pos, (scores.shape[0],), "pos")
    _shape(topk, (scores.shape[0], k), "topk")
    _check(_lib().dsa_topk_select(_ptr(scores), scores.shape[1], _ptr(pos), pos.numel(), k,
                                  max_ctx, _ptr(topk), _stream(stream)))


def dsa_indexer_topk(q_idx, w, k_idx, cu, n_req, pos, bid, k, max_ctx, topk, workspace,
                     block_table=None, page_size=64, stream=None):
    """Indexer scores + top-k; the score rows live in `workspace` (uint8, 256-byte aligned)."""
    _dev(q_idx, torch.bfloat16, "q_idx"); _dev(k_idx, torch.bfloat16, "k_idx")
    _dev(w, torch.float32, "w"); _dev(topk, torch.int32, "topk")
    _dev(pos, torch.int32, "pos"); _dev(bid, torch.int32, "bid"); _dev(cu, torch.int32, "cu")
    _dev(block_table, torch.int32, "block_table")
    n_q, Hi, Di = q_idx.shape
    _indexer_shapes(q_idx, w, pos, bid, block_table, n_req)
    _shape(topk, (n_q, k), "topk")
    max_pages = block_table.shape[1] if block_table is not None else 0
    _check(_lib().dsa_indexer_topk(
        _ptr(q_idx), _ptr(w), _ptr(k_idx), k_idx.shape[0], _ptr(cu), n_req, _ptr(pos), _ptr(bid),
        n_q, Hi, Di, k, max_ctx, _ptr(block_table), max_pages, page_size, _ptr(topk),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def dsa_indexer_topk_noalloc(q_idx, w, k_idx, cu, n_req, pos, bid, k, max_ctx, topk,
                             block_table=None, page_size=64, stream=None):
    """dsa_indexer_topk without a workspace argument: for callers that cannot allocate device
    memory; the library's static scratch array is used instead (calls must not overlap)."""
    _dev(q_idx, torch.bfloat16, "q_idx"); _dev(k_idx, torch.bfloat16, "k_idx")
    _dev(w, torch.float32, "w"); _dev(topk, torch.int32, "topk")
    _dev(pos, torch.int32, "pos"); _dev(bid, torch.int32, "bid"); _dev(cu, torch.int32, "cu")
    _dev(block_table, torch.int32, "block_table")
    n_q, Hi, Di = q_idx.shape
    _indexer_shapes(q_idx, w, pos, bid, block_table, n_req)
    _shape(topk, (n_q, k), "topk")
    max_pages = block_table.shape[1] if block_table is not None else 0
    _check(_lib().dsa_indexer_topk_noalloc(
        _ptr(q_idx), _ptr(w), _ptr(k_idx), k_idx.shape[0], _ptr(cu), n_req, _ptr(pos), _ptr(bid),
        n_q, Hi, Di, k, max_ctx, _ptr(block_table), max_pages, page_size, _ptr(topk),
        _stream(stream)))


def dsa_quantize_fp8_rows(x, codes, scales, stream=None):
    """x bf16 [rows, 128] -> codes uint8 [rows, 128] (E4M3), scales fp32 [rows]; x may be any
    shape whose last dimension is 128 (q_idx [n_q, Hi, 128] gives scales [n_q, Hi])."""
    _dev(x, torch.bfloat16, "x"); _dev(codes, torch.uint8, "codes"); _dev(scales, torch.float32, "scales")
    cols = x.shape[-1]
    rows = x.numel() // cols if cols else 0
    if codes.shape != x.shape or scales.numel() != rows:
        raise ValueError("codes must match x's shape and scales hold one value per row")
    _check(_lib().dsa_quantize_fp8_rows(_ptr(x), rows, cols, _ptr(codes), _ptr(scales),
                                        _stream(stream)))


FP8_LATENT_ROW_BYTES = 656


def _latent_pair(c, packed):
    _dev(c, torch.bfloat16, "c"); _dev(packed, torch.uint8, "packed")
    if c.dim() != 2 or c.shape[1] != 576:
        raise ValueError(f"c must be [rows, 576], got {tuple(c.shape)}")
    _shape(packed, (c.shape[0], FP8_LATENT_ROW_BYTES), "packed")
    return c.shape[0]


def dsa_quantize_fp8_latent(c, packed, stream=None):
    """c bf16 [rows, 576] -> packed uint8 [rows, 656]: 512 E4M3 codes, 4 fp32 block scales,
    64 bf16 rope values."""
    rows = _latent_pair(c, packed)
    _check(_lib().dsa_quantize_fp8_latent(_ptr(c), rows, _ptr(packed), _stream(stream)))


def dsa_dequantize_fp8_latent(packed, c, stream=None):
    """packed uint8 [rows, 656] -> c bf16 [rows, 576], the rows the sparse MLA reads."""
    rows = _latent_pair(c, packed)
    _check(_lib().dsa_dequantize_fp8_latent(_ptr(packed), rows, _ptr(c), _stream(stream)))


def _fp8_indexer_checks(q8, q_scale, w, k8, k_scale, pos, bid, block_table, n_req):
    _dev(q8, torch.uint8, "q8"); _dev(k8, torch.uint8, "k8")
    _dev(q_scale, torch.float32, "q_scale"); _dev(k_scale, torch.float32, "k_scale")
    _dev(w, torch.float32, "w"); _dev(pos, torch.int32, "pos"); _dev(bid, torch.int32, "bid")
    _dev(block_table, torch.int32, "block_table")
    n_q, Hi, _ = q8.shape
    _shape(q_scale, (n_q, Hi), "q_scale")
    _shape(k_scale, (k8.shape[0],), "k_scale")
    _indexer_shapes(q8, w, pos, bid, block_table, n_req)


def dsa_indexer_scores_fp8(q8, q_scale, w, k8, k_scale, cu, n_req, pos, bid, max_ctx, scores,
                           workspace, block_table=None, page_size=64, stream=None):
    """Indexer scores on E4M3 rows: the indexer of (q_scale q8, k_scale k8)."""
    _fp8_indexer_checks(q8, q_scale, w, k8, k_scale, pos, bid, block_table, n_req)
    _dev(scores, torch.float32, "scores"); _dev(cu, torch.int32, "cu")
    n_q, Hi, Di = q8.shape
    _shape(scores, (n_q, None), "scores")
    max_pages = block_table.shape[1] if block_table is not None else 0
    _check(_lib().dsa_indexer_scores_fp8(
        _ptr(q8), _ptr(q_scale), _ptr(w), _ptr(k8), _ptr(k_scale), k8.shape[0], _ptr(cu), n_req,
        _ptr(pos), _ptr(bid), n_q, Hi, Di, max_ctx, _ptr(block_table), max_pages, page_size,
        _ptr(scores), scores.shape[1], _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def dsa_indexer_topk_fp8(q8, q_scale, w, k8, k_scale, cu, n_req, pos, bid, k, max_ctx, topk,
                         workspace, block_table=None, page_size=64, stream=None):
    """dsa_indexer_topk on E4M3 rows (same workspace size, same selection rule)."""
    _fp8_indexer_checks(q8, q_scale, w, k8, k_scale, pos, bid, block_table, n_req)
    _dev(topk, torch.int32, "topk"); _dev(cu, torch.int32, "cu")
    n_q, Hi, Di = q8.shape
    _shape(topk, (n_q, k), "topk")
    max_pages = block_table.shape[1] if block_table is not None else 0
    _check(_lib().dsa_indexer_topk_fp8(
        _ptr(q8), _ptr(q_scale), _ptr(w), _ptr(k8), _ptr(k_scale), k8.shape[0], _ptr(cu), n_req,
        _ptr(pos), _ptr(bid), n_q, Hi, Di, k, max_ctx, _ptr(block_table), max_pages, page_size,
        _ptr(topk), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def dsa_sparse_mla(q, c, cu, n_req, bid, topk, scale, o, lse=None, block_table=None,
                   page_size=64, stream=None):
    """o[t,h] = softmax(scale q[t,h] . c[rows]) c[rows, :dv] over the valid top-k rows."""
    _dev(q, torch.bfloat16, "q"); _dev(c, torch.bfloat16, "c"); _dev(o, torch.bfloat16, "o")
    _dev(bid, torch.int32, "bid"); _dev(topk, torch.int32, "topk"); _dev(cu, torch.int32, "cu")
    _dev(lse, torch.float32, "lse"); _dev(block_table, torch.int32, "block_table")
    n_q, H, dqk = q.shape
    dv = o.shape[2]
    _mla_shapes(q, c, o, lse, bid, None, topk, block_table, n_req)
    max_pages = block_table.shape[1] if block_table is not None else 0
    _check(_lib().dsa_sparse_mla(
        _ptr(q), _ptr(c), c.shape[0], _ptr(cu), n_req, _ptr(bid), _ptr(topk), n_q, H, dqk, dv,
        topk.shape[1], float(scale), _ptr(block_table), max_pages, page_size, _ptr(o), _ptr(lse),
        _stream(stream)))


def _mla_shapes(q, c, o, lse, bid, pos, topk, block_table, n_req):
    n_q, H, dqk = q.shape
    _shape(c, (None, dqk), "c")
    _shape(o, (n_q, H, None), "o")
    _shape(lse, (n_q, H), "lse")
    _shape(bid, (n_q,), "bid")
    _shape(pos, (n_q,), "pos")
    _shape(topk, (n_q, None), "topk")
    _shape(block_table, (n_req, None), "block_table")


def dsa_sparse_mla_workspace_size(n_q: int) -> int:
    return int(_lib().dsa_sparse_mla_workspace_size(n_q))


def dsa_sparse_mla_balanced(q, c, cu, n_req, bid, pos, topk, scale, o, workspace, lse=None,
                            block_table=None, page_size=64, stream=None):
    """dsa_sparse_mla with the persistent pairs' work ordered by min(pos + 1, k) (same result)."""
    _dev(q, torch.bfloat16, "q"); _dev(c, torch.bfloat16, "c"); _dev(o, torch.bfloat16, "o")
    _dev(bid, torch.int32, "bid"); _dev(pos, torch.int32, "pos"); _dev(topk, torch.int32, "topk")
    _dev(cu, torch.int32, "cu"); _dev(lse, torch.float32, "lse")
    _dev(block_table, torch.int32, "block_table")
    if workspace is None:
        raise ValueError("workspace is required (dsa_sparse_mla_workspace_size bytes)")
    _dev(workspace, None, "workspace")
    n_q, H, dqk = q.shape
    dv = o.shape[2]
    _mla_shapes(q, c, o, lse, bid, pos, topk, block_table, n_req)
    max_pages = block_table.shape[1] if block_table is not None else 0
    _check(_lib().dsa_sparse_mla_balanced(
        _ptr(q), _ptr(c), c.shape[0], _ptr(cu), n_req, _ptr(bid), _ptr(pos), _ptr(topk), n_q, H,
        dqk, dv, topk.shape[1], float(scale), _ptr(block_table), max_pages, page_size, _ptr(o),
        _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))
