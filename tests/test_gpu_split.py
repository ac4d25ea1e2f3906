"""GPU parity: round-robin split metadata, row gather and rerange vs the oracle (bit-exact)."""
import numpy as np
import pytest
import torch

import workloads as W
from dsa_cases import gpu_gather_and_rerange, gpu_split
from oracle import rerange as orr
from oracle import split as osplit

pytestmark = pytest.mark.gpu


def _cases():
    out = [(W.cu_seqlens(W.WORKLOADS[i].lengths), W.WORKLOADS[i].sp) for i in (0, 1, 2, 3)]
    rng = np.random.default_rng(5)
    out.append((np.array([0, 0], np.int32), 4))                 # empty batch
    out.append((np.array([0, 3], np.int32), 8))                 # fewer tokens than shards
    out.append((np.array([0, 0, 5, 5, 9, 9], np.int32), 3))     # empty requests
    out.append((W.cu_seqlens([1000]), 1))                       # sp = 1
    for _ in range(4):
        L = rng.integers(0, 400, int(rng.integers(1, 12)))
        out.append((W.cu_seqlens(L), int(rng.integers(1, 17))))
    return out


@pytest.mark.parametrize("case", range(12))
def test_split_metadata_matches_oracle(case):
    cu, sp = _cases()[case]
    for r in range(sp):
        g = gpu_split(cu, sp, r)
        o = osplit.round_robin_split(cu, sp, r)
        for key in ("gidx", "bid", "pos", "cu_shard"):
            assert np.array_equal(g[key], o[key]), (case, r, key)


@pytest.mark.parametrize("wid", [0, 1, 2, 3])
@pytest.mark.parametrize("padded", [False, True])
@pytest.mark.parametrize("width", [576, 128, 328])     # latent rows (1152 B), k_idx rows (256 B), FP8 latent rows (656 B)
def test_gather_and_rerange_workloads(wid, padded, width):
    wl = W.WORKLOADS[wid]
    cu = W.cu_seqlens(wl.lengths)
    n = int(cu[-1])
    g = torch.Generator(device="cuda").manual_seed(17 + wid)
    logical = torch.randint(-32768, 32767, (n, width), generator=g, device="cuda",
                            dtype=torch.int32).to(torch.int16)
    gathered, out = gpu_gather_and_rerange(logical, cu, wl.sp, padded)
    x = logical.cpu().numpy()
    stride = (-(-n // wl.sp)) if padded else 0
    ora_gathered = orr.all_gather([osplit.split_rows(x, wl.sp, r) for r in range(wl.sp)], stride)
    assert np.array_equal(gathered.cpu().numpy(), ora_gathered)
    assert np.array_equal(out.cpu().numpy(), x)
    assert np.array_equal(orr.rerange(ora_gathered, n, wl.sp, stride), x)


@pytest.mark.parametrize("row_bytes", [1, 6, 20, 1152])
def test_rerange_of_oracle_gather_odd_rows(row_bytes):
    """Rows that are not 16-byte multiples take the byte path; the input is the oracle's."""
    rng = np.random.default_rng(row_bytes)
    n, sp = 1003, 6
    x = rng.integers(0, 256, (n, row_bytes), dtype=np.uint8)
    gathered = orr.all_gather([osplit.split_rows(x, sp, r) for r in range(sp)])
    out = torch.empty((n, row_bytes), dtype=torch.uint8, device="cuda")
    import deepseek_v3_sparse_round_gb300 as dsa
    dsa.dsa_rr_rerange(torch.as_tensor(gathered).cuda(), out, n, sp, 0)
    assert np.array_equal(out.cpu().numpy(), x)


def _paged_case(lengths, sp, ps, seed, width, dtype=torch.bfloat16, spare_pages=3):
    """Logical rows x (seeded), the rank-major gathered buffer, a random block table and a pool
    pre-filled with a sentinel."""
    rng = np.random.default_rng(seed)
    cu = W.cu_seqlens(lengths)
    n = int(cu[-1])
    need = [-(-int(L) // ps) for L in lengths]
    n_pages = sum(need) + spare_pages
    perm = rng.permutation(n_pages)
    table = np.full((len(lengths), max(max(need), 1)), -1, dtype=np.int32)
    at = 0
    for b, p in enumerate(need):
        table[b, :p] = perm[at:at + p]
        at += p
    x = W.normal_bf16((n, width), seed=seed, device="cuda") if dtype == torch.bfloat16 \
        else W.int_uniform((n, width), 0, 254, seed, dtype=torch.uint8, device="cuda")
    pool0 = torch.full((n_pages * ps, width), 7, dtype=x.dtype, device="cuda")
    return cu, n, table, x, pool0


def _oracle_pool(gathered, cu, sp, stride, table, ps, pool0):
    g = gathered.cpu().view(torch.uint8).numpy() if gathered.dtype == torch.bfloat16 else gathered.cpu().numpy()
    p = pool0.cpu().view(torch.uint8).numpy() if pool0.dtype == torch.bfloat16 else pool0.cpu().numpy()
    return orr.rerange_into_pages(g, cu, sp, stride, table, ps, p)


@pytest.mark.parametrize("wid", [1, 3])
@pytest.mark.parametrize("padded", [False, True])
@pytest.mark.parametrize("width", [576, 128, 328])   # 328 bf16 = 656 B, a packed FP8 latent row
def test_rerange_paged_workloads(wid, padded, width):
    from dsa_cases import dsa, i32
    wl = W.WORKLOADS[wid]
    cu, n, table, x, pool0 = _paged_case(wl.lengths, wl.sp, 64, 11 + wid, width)
    gathered, _ = gpu_gather_and_rerange(x, cu, wl.sp, padded)
    stride = (-(-n // wl.sp)) if padded else 0
    pool = pool0.clone()
    dsa().dsa_rr_rerange_paged(gathered, pool, n, wl.sp, i32(cu), i32(table), stride, 64)
    want = _oracle_pool(gathered, cu, wl.sp, stride, table, 64, pool0)
    got = pool.cpu().view(torch.uint8).numpy()
    assert np.array_equal(got, want)
    assert dsa().dsa_read_device_errors() == 0


@pytest.mark.parametrize("seed", range(4))
def test_rerange_paged_edge_cases(seed):
    """Odd page sizes, empty requests, byte rows (row size not a multiple of 16), sp = 1."""
    from dsa_cases import dsa, i32
    rng = np.random.default_rng(seed)
    lengths = [int(v) for v in rng.integers(0, 300, int(rng.integers(1, 9)))]
    lengths[0] = 0
    sp = int(rng.integers(1, 9))
    ps = int(rng.choice([1, 3, 16, 64]))
    width = int(rng.choice([7, 32]))                       # 7-byte rows: byte path
    cu, n, table, x, pool0 = _paged_case(lengths, sp, ps, 50 + seed, width, dtype=torch.uint8)
    shards = [gpu_split(cu, sp, r, src=x)["rows"] for r in range(sp)]
    gathered = torch.cat(shards)
    pool = pool0.clone()
    dsa().dsa_rr_rerange_paged(gathered, pool, n, sp, i32(cu), i32(table), 0, ps)
    want = orr.rerange_into_pages(gathered.cpu().numpy(), cu, sp, 0, table, ps, pool0.cpu().numpy())
    assert np.array_equal(pool.cpu().numpy(), want)
    assert dsa().dsa_read_device_errors() == 0


def test_rerange_paged_missing_page_is_skipped_and_flagged():
    from dsa_cases import dsa, i32
    lengths = [130, 70]
    cu, n, table, x, pool0 = _paged_case(lengths, 4, 64, 3, 128)
    table = table.copy()
    lost = int(table[0, 1])
    table[0, 1] = -1                                       # request 0, positions 64..127
    gathered, _ = gpu_gather_and_rerange(x, cu, 4, False)
    pool = pool0.clone()
    dsa().dsa_rr_rerange_paged(gathered, pool, n, 4, i32(cu), i32(table), 0, 64)
    assert dsa().dsa_read_device_errors() & dsa().DEVERR_BAD_INDEX
    got = pool.cpu()
    assert torch.equal(got[lost * 64:(lost + 1) * 64], pool0.cpu()[lost * 64:(lost + 1) * 64])
    keep = table.copy()
    keep[0, 1] = lost
    kv_rows = [int(keep[0, 0]) * 64 + s for s in range(64)] + [int(keep[1, 0]) * 64 + s for s in range(64)]
    src_rows = list(range(64)) + [130 + s for s in range(64)]
    assert torch.equal(got[kv_rows], x.cpu()[src_rows])


def _local_table(cu, sp, r, ps, seed, spare=2):
    """Rank r's own block table: request b needs ceil(cnt_b / ps) pages, cnt_b = its tokens on
    the rank (counted from the oracle's token list); page ids a seeded permutation."""
    rng = np.random.default_rng(seed)
    tokens = osplit.shard_tokens(int(cu[-1]), sp, r)
    counts = [int(np.sum((tokens >= cu[b]) & (tokens < cu[b + 1]))) for b in range(len(cu) - 1)]
    need = [-(-c // ps) for c in counts]
    perm = rng.permutation(sum(need) + spare)
    table = np.full((len(counts), max(max(need), 1)), -1, dtype=np.int32)
    at = 0
    for b, p in enumerate(need):
        table[b, :p] = perm[at:at + p]
        at += p
    return table, sum(need) + spare


@pytest.mark.parametrize("wid", [1, 3])
@pytest.mark.parametrize("width", [576, 128, 328])   # 328 bf16 = 656 B, a packed FP8 latent row
def test_cache_local_paged_workloads(wid, width):
    """Every rank keeps only its own tokens: bit-exact against the oracle for each shard, with
    the rank's rows coming from the split's gather (as a rank holds them after step A)."""
    from dsa_cases import dsa, i32
    wl = W.WORKLOADS[wid]
    cu = W.cu_seqlens(wl.lengths)
    n = int(cu[-1])
    x = W.normal_bf16((n, width), seed=70 + wid, device="cuda")
    for r in range(wl.sp):
        local = gpu_split(cu, wl.sp, r, src=x)["rows"]
        table, n_pages = _local_table(cu, wl.sp, r, 64, 90 + r)
        pool0 = torch.full((n_pages * 64, width), 3, dtype=torch.bfloat16, device="cuda")
        pool = pool0.clone()
        dsa().dsa_rr_cache_local_paged(local, pool, n, wl.sp, r, i32(cu), i32(table), 64)
        want = orr.cache_local_into_pages(local.cpu().view(torch.uint8).numpy(), cu, wl.sp, r,
                                          table, 64, pool0.cpu().view(torch.uint8).numpy())
        assert np.array_equal(pool.cpu().view(torch.uint8).numpy(), want), r
    assert dsa().dsa_read_device_errors() == 0


@pytest.mark.parametrize("seed", range(4))
def test_cache_local_paged_edge_cases(seed):
    """Empty requests, requests with no token on the rank, odd page sizes, byte rows."""
    from dsa_cases import dsa, i32
    rng = np.random.default_rng(300 + seed)
    lengths = [int(v) for v in rng.integers(0, 40, int(rng.integers(1, 9)))]
    lengths[0] = 0
    sp = int(rng.integers(1, 9))
    ps = int(rng.choice([1, 3, 16, 64]))
    width = int(rng.choice([7, 32]))
    cu = W.cu_seqlens(lengths)
    n = int(cu[-1])
    x = W.int_uniform((max(n, 1), width), 0, 254, 60 + seed, dtype=torch.uint8, device="cuda")[:n]
    for r in range(sp):
        n_r = dsa().dsa_rr_shard_len(n, sp, r)
        local = x[r::sp].contiguous() if n_r else torch.empty((0, width), dtype=torch.uint8, device="cuda")
        table, n_pages = _local_table(cu, sp, r, ps, 400 + r)
        pool0 = torch.full((n_pages * ps, width), 9, dtype=torch.uint8, device="cuda")
        pool = pool0.clone()
        dsa().dsa_rr_cache_local_paged(local, pool, n, sp, r, i32(cu), i32(table), ps)
        want = orr.cache_local_into_pages(local.cpu().numpy(), cu, sp, r, table, ps,
                                          pool0.cpu().numpy())
        assert np.array_equal(pool.cpu().numpy(), want), (r, sp, ps)
    assert dsa().dsa_read_device_errors() == 0


def test_cache_local_paged_missing_page_is_skipped_and_flagged():
    from dsa_cases import dsa, i32
    cu = W.cu_seqlens([600, 90])
    sp, r = 4, 1
    x = W.normal_bf16((690, 128), seed=8, device="cuda")
    local = gpu_split(cu, sp, r, src=x)["rows"]
    table, n_pages = _local_table(cu, sp, r, 64, 5)
    lost = int(table[0, 1])
    bad = table.copy()
    bad[0, 1] = -1                                   # request 0, rank-local slots 64..127
    pool0 = torch.full((n_pages * 64, 128), 3, dtype=torch.bfloat16, device="cuda")
    pool = pool0.clone()
    dsa().dsa_rr_cache_local_paged(local, pool, 690, sp, r, i32(cu), i32(bad), 64)
    assert dsa().dsa_read_device_errors() & dsa().DEVERR_BAD_INDEX
    assert torch.equal(pool[lost * 64:(lost + 1) * 64], pool0[lost * 64:(lost + 1) * 64])
    want = orr.cache_local_into_pages(local.cpu().view(torch.uint8).numpy(), cu, sp, r, table, 64,
                                      pool0.cpu().view(torch.uint8).numpy())
    got = pool.cpu().view(torch.uint8).numpy()
    keep = np.ones(len(got), bool)
    keep[lost * 64:(lost + 1) * 64] = False
    assert np.array_equal(got[keep], want[keep])


@pytest.mark.parametrize("wid", [0, 1, 2, 3])
@pytest.mark.parametrize("padded", [False, True])
def test_rerange_multi_matches_oracle(wid, padded):
    """k_idx rows (256 B) and latent rows (1152 B) of the same tokens reranged by one launch:
    each bit-exact against the oracle's rerange of the oracle's all-gather layout."""
    from dsa_cases import dsa
    wl = W.WORKLOADS[wid]
    cu = W.cu_seqlens(wl.lengths)
    n = int(cu[-1])
    stride = (-(-n // wl.sp)) if padded else 0
    xs = [W.int_uniform((n, width), -32768, 32767, 40 + width, dtype=torch.int32,
                        device="cuda").to(torch.int16) for width in (128, 576, 8)]
    gathered = []
    for x in xs:
        g = orr.all_gather([osplit.split_rows(x.cpu().numpy(), wl.sp, r) for r in range(wl.sp)],
                           stride)
        gathered.append(torch.as_tensor(g).cuda())
    outs = [torch.full_like(x, 7) for x in xs]
    dsa().dsa_rr_rerange_multi(gathered, outs, n, wl.sp, stride)
    for x, g, o in zip(xs, gathered, outs):
        assert np.array_equal(o.cpu().numpy(), orr.rerange(g.cpu().numpy(), n, wl.sp, stride))
        assert torch.equal(o, x)


def test_rerange_multi_rejects_unaligned_rows():
    from dsa_cases import dsa
    a = torch.zeros((10, 3), dtype=torch.uint8, device="cuda")     # 3-byte rows
    with pytest.raises(dsa().DsaError):
        dsa().dsa_rr_rerange_multi([a], [torch.empty_like(a)], 10, 2)
