"""Seeded synthetic inputs for the round-robin sequence-shard DSA attention path.

This module only draws random numbers and lays them out. It holds none of the method's
arithmetic (no split, rerange, score, selection or attention), so both the CUDA path
(tests, bench) and the fp64 oracle (tests) can take their inputs from it without sharing
any computation.

Five workloads, in order:

  0 "tiny"       1 request of 256 tokens, sp=4, shard rank 1 (64 queries). Indexer 4 heads x 32,
                 q_idx / k_idx integers U[-3,3], w integers U[0,3]; top-k 32. MLA 8 heads,
                 qk dim 80 (64 latent + 16 rope), v dim 64, q and kv N(0,1)/sqrt(80). Seed 0.
  1 "varlen"     4 requests {8000, 800, 5, 3000}, sp=8, shard rank 3 (1,476 queries). Indexer
                 64 x 128 bf16 N(0,1), w N(0,1)/8, top-k 2048. MLA 128 heads, 576/512, bf16
                 N(0,1), scale 1/sqrt(576).
  2 "long"       1 request of 32,768 tokens, sp=8, all 8 shards (4,096 queries each).
  3 "many_req"   32 requests with lengths U[128, 4096] (seed 0 -> N = 71,014), sp=4, all shards.
  4 "decode"     64 requests, 2 new query tokens each, context U[16384, 65536], KV in 64-token
                 pages under a random block table (sp=1, no split).

Values are drawn with torch generators (CPU for the small workloads, the current CUDA device
for the large ones) so that multi-gigabyte query tensors are made where they are used.
Integer-valued indexer inputs (q_idx, k_idx, w in [-3, 3]) make every score exact in fp32 and
are used wherever index sets must match bit for bit.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    lengths: tuple          # request lengths (tokens); for "decode", the context lengths
    sp: int                 # number of sequence shards
    ranks: tuple            # shard ranks processed
    Hi: int                 # indexer heads
    Di: int                 # indexer head dim
    topk: int               # k of the per-query top-k
    H: int                  # MLA heads
    dc: int                 # latent (kv_lora) width
    dr: int                 # rope width
    dv: int                 # value width (first dv columns of the latent row)
    seed: int = 0
    integer_indexer: bool = False   # workload 0 draws integer indexer inputs
    mla_std: float = 1.0            # std of q / kv values
    w_std: float = 1.0 / 8.0        # std of the indexer head weights (non-integer case)
    decode_queries: int = 0         # >0: decode workload, queries per request at the context end
    page_size: int = 0              # >0: KV lives in pages of this many tokens

    @property
    def dqk(self) -> int:
        return self.dc + self.dr

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.dqk)

    @property
    def n_tokens(self) -> int:
        return int(sum(self.lengths))


def _many_req_lengths() -> tuple:
    rng = np.random.default_rng(0)
    return tuple(int(x) for x in rng.integers(128, 4097, 32))


def _decode_ctx_lengths() -> tuple:
    rng = np.random.default_rng(0)
    return tuple(int(x) for x in rng.integers(16384, 65537, 64))


WORKLOADS = {
    0: Workload("tiny", (256,), 4, (1,), Hi=4, Di=32, topk=32, H=8, dc=64, dr=16, dv=64,
                integer_indexer=True, mla_std=1.0 / math.sqrt(80.0)),
    1: Workload("varlen", (8000, 800, 5, 3000), 8, (3,), Hi=64, Di=128, topk=2048,
                H=128, dc=512, dr=64, dv=512),
    2: Workload("long", (32768,), 8, tuple(range(8)), Hi=64, Di=128, topk=2048,
                H=128, dc=512, dr=64, dv=512),
    3: Workload("many_req", _many_req_lengths(), 4, tuple(range(4)), Hi=64, Di=128,
                topk=2048, H=128, dc=512, dr=64, dv=512),
    4: Workload("decode", _decode_ctx_lengths(), 1, (0,), Hi=64, Di=128, topk=2048,
                H=128, dc=512, dr=64, dv=512, decode_queries=2, page_size=64),
}


def cu_seqlens(lengths) -> np.ndarray:
    """Exclusive prefix offsets [0, L0, L0+L1, ...] (int32) of a varlen batch."""
    out = np.zeros(len(lengths) + 1, dtype=np.int64)
    out[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return out.astype(np.int32)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, seed: int, std: float = 1.0, device="cpu") -> torch.Tensor:
    """N(0, std^2) values drawn in fp32 and rounded once to bf16 (round to nearest even)."""
    x = torch.randn(*shape, generator=_gen(seed, device), device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def normal_f32(shape, seed: int, std: float = 1.0, device="cpu") -> torch.Tensor:
    x = torch.randn(*shape, generator=_gen(seed, device), device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x


def int_uniform(shape, lo: int, hi: int, seed: int, dtype=torch.bfloat16, device="cpu"):
    """Integers uniform in [lo, hi] (inclusive), stored exactly in `dtype`."""
    x = torch.randint(lo, hi + 1, tuple(shape), generator=_gen(seed, device), device=device)
    return x.to(dtype)


def seed_of(wl: Workload, what: str, rank: int = 0) -> int:
    """A distinct, fixed seed per (workload, tensor, shard) so draws never alias."""
    order = ("q_idx", "k_idx", "w", "q", "c", "block_table", "gathered_pad", "rows")
    return wl.seed * 1_000_003 + (order.index(what) + 1) * 10_007 + rank * 101


@dataclass
class IndexerInputs:
    q_idx: torch.Tensor     # bf16 [n_q, Hi, Di]
    w: torch.Tensor         # fp32 [n_q, Hi]
    k_idx: torch.Tensor     # bf16 [n_kv_rows, Di]


@dataclass
class MlaInputs:
    q: torch.Tensor         # bf16 [n_q, H, dqk]
    c: torch.Tensor         # bf16 [n_kv_rows, dqk]


def indexer_inputs(wl: Workload, n_q: int, n_kv_rows: int, rank: int, integer: bool = None,
                   device="cpu") -> IndexerInputs:
    integer = wl.integer_indexer if integer is None else integer
    if integer:
        w_lo = 0 if wl.integer_indexer else -3
        q_idx = int_uniform((n_q, wl.Hi, wl.Di), -3, 3, seed_of(wl, "q_idx", rank), device=device)
        k_idx = int_uniform((n_kv_rows, wl.Di), -3, 3, seed_of(wl, "k_idx"), device=device)
        w = int_uniform((n_q, wl.Hi), w_lo, 3, seed_of(wl, "w", rank), dtype=torch.float32,
                        device=device)
    else:
        q_idx = normal_bf16((n_q, wl.Hi, wl.Di), seed_of(wl, "q_idx", rank), device=device)
        k_idx = normal_bf16((n_kv_rows, wl.Di), seed_of(wl, "k_idx"), device=device)
        w = normal_f32((n_q, wl.Hi), seed_of(wl, "w", rank), std=wl.w_std, device=device)
    return IndexerInputs(q_idx, w, k_idx)


def mla_inputs(wl: Workload, n_q: int, n_kv_rows: int, rank: int, device="cpu") -> MlaInputs:
    q = normal_bf16((n_q, wl.H, wl.dqk), seed_of(wl, "q", rank), std=wl.mla_std, device=device)
    c = normal_bf16((n_kv_rows, wl.dqk), seed_of(wl, "c"), std=wl.mla_std, device=device)
    return MlaInputs(q, c)


def random_block_table(ctx_lengths, page_size: int, seed: int):
    """A random page assignment for a paged KV pool.

    Request b needs ceil(C_b / page_size) pages; the physical page ids of all requests are a
    seeded random permutation of 0..total_pages-1. Returns (block_table int32 [B, max_pages],
    padded with -1, total_pages).
    """
    pages = [(int(c) + page_size - 1) // page_size for c in ctx_lengths]
    total = int(sum(pages))
    perm = np.random.default_rng(seed).permutation(total).astype(np.int32)
    max_pages = max(pages) if pages else 0
    table = np.full((len(pages), max(max_pages, 1)), -1, dtype=np.int32)
    at = 0
    for b, p in enumerate(pages):
        table[b, :p] = perm[at:at + p]
        at += p
    return table, total


def decode_queries(ctx_lengths, per_request: int):
    """Batch ids and positions of decode queries: the last `per_request` tokens of each context."""
    bid, pos = [], []
    for b, c in enumerate(ctx_lengths):
        for j in range(per_request):
            bid.append(b)
            pos.append(int(c) - per_request + j)
    return np.asarray(bid, dtype=np.int32), np.asarray(pos, dtype=np.int32)


def random_lengths(n: int, lo: int, hi: int, seed: int) -> tuple:
    rng = np.random.default_rng(seed)
    return tuple(int(x) for x in rng.integers(lo, hi + 1, n))


def sample_queries(n_q: int, must: np.ndarray, n_sample: int, seed: int) -> np.ndarray:
    """Sorted unique query indices: every index in `must` plus random others up to n_sample."""
    rng = np.random.default_rng(seed)
    must = np.unique(np.asarray(must, dtype=np.int64))
    rest = np.setdiff1d(np.arange(n_q), must)
    extra = max(0, n_sample - len(must))
    pick = rng.choice(rest, size=min(extra, len(rest)), replace=False) if len(rest) else rest
    return np.unique(np.concatenate([must, pick]))


# E4M3 byte codes of the small integers -3..3 (sign bit 0x80; 1 = 0x38, 2 = 0x40, 3 = 0x44 under
# the E4M3 layout: 4 exponent bits with bias 7, 3 mantissa bits). Input layout only: the tests
# use them to build FP8 rows whose values are exact integers.
_E4M3_SMALL_INT_CODES = {-3: 0xC4, -2: 0xC0, -1: 0xB8, 0: 0x00, 1: 0x38, 2: 0x40, 3: 0x44}


def int_codes_e4m3(shape, lo: int, hi: int, seed: int, device="cpu") -> torch.Tensor:
    """uint8 E4M3 codes of integers uniform in [lo, hi] (within -3..3)."""
    assert -3 <= lo <= hi <= 3
    table = torch.zeros(7, dtype=torch.uint8)
    for v, c in _E4M3_SMALL_INT_CODES.items():
        table[v + 3] = c
    x = torch.randint(lo, hi + 1, tuple(shape), generator=_gen(seed, device), device=device)
    return table.to(device)[x + 3]


def pow2_scales(shape, lo_exp: int, hi_exp: int, seed: int, device="cpu") -> torch.Tensor:
    """fp32 powers of two 2^e with e uniform in [lo_exp, hi_exp]."""
    e = torch.randint(lo_exp, hi_exp + 1, tuple(shape), generator=_gen(seed, device), device=device)
    return torch.pow(2.0, e.to(torch.float32))
