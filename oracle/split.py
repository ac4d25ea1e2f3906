"""Oracle: round-robin split of a flattened varlen batch.

Test infrastructure only (see the package docstring).

Source: "[DeepSeek v3.2] 上下文并行详解", section 2.B (nsa_cp_round_robin_split_data): rank
`cp_rank` keeps the rows `arange(cp_rank, tokens, cp_size)` of the flattened input, and a
metadata kernel recomputes the per-rank cu_seqlens and batch indices after the scatter;
section 4 part 1 asks for the mapping "rank X's token <-> batch Y logical position Z"; section 4
part 3 step 1 works the example of 8 tokens on 4 ranks.

Reading taken where the page is silent: the round-robin index is the token's index g in the
flattened batch (the code slices the whole `input_`), so a request with no token on a rank
keeps a zero-length entry in that rank's cu_seqlens.
"""
from __future__ import annotations

import numpy as np


def shard_tokens(n_tokens: int, sp: int, rank: int) -> np.ndarray:
    """Flattened indices g that rank `rank` of `sp` keeps: rank, rank+sp, rank+2sp, ... < N."""
    return np.arange(rank, n_tokens, sp, dtype=np.int64)


def round_robin_split(cu, sp: int, rank: int) -> dict:
    """Shard metadata for one rank.

    cu: request offsets [B+1] (cu[0] = 0, cu[B] = N). Returns int64 arrays:
      gidx     [n_r]  flattened token index of each shard token, ascending
      bid      [n_r]  request of each shard token: the largest b with cu[b] <= g
      pos      [n_r]  logical position inside its request: g - cu[bid]
      cu_shard [B+1]  offsets of each request's tokens inside the shard
    """
    cu = np.asarray(cu, dtype=np.int64)
    n_req = len(cu) - 1
    gidx = shard_tokens(int(cu[-1]), sp, rank)
    bid = np.searchsorted(cu, gidx, side="right") - 1
    pos = gidx - cu[bid]
    per_req = np.bincount(bid, minlength=n_req) if n_req > 0 else np.zeros(0, np.int64)
    cu_shard = np.zeros(n_req + 1, dtype=np.int64)
    cu_shard[1:] = np.cumsum(per_req)
    return {"gidx": gidx, "bid": bid, "pos": pos, "cu_shard": cu_shard}


def split_rows(src: np.ndarray, sp: int, rank: int) -> np.ndarray:
    """The rank's rows of a per-token tensor: src[arange(rank, N, sp)] (section 2.B)."""
    return src[shard_tokens(src.shape[0], sp, rank)]


def round_robin_split_decode(cu_new, pos_base, sp: int, rank: int) -> dict:
    """Round-robin split of a decode step's new tokens ("[RFC]: Parallel strategy for Deepseek
    v3.2 like models", "New proposal": sequence parallel over the token dimension for both
    prefill and decode). The flattened batch is the new tokens only (cu_new); a new token's
    logical position is its request's earlier context pos_base[b] plus its index among the
    request's new tokens. Reading: the same dealing as prefill (section 2.B of "[DeepSeek v3.2]
    上下文并行详解"), applied to the decode batch."""
    out = round_robin_split(cu_new, sp, rank)
    base = np.asarray(pos_base, dtype=np.int64)
    out["pos"] = out["pos"] + base[out["bid"]]
    return out
