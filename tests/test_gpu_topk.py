"""GPU parity: radix-select top-k on fp32 score rows vs the oracle's full sort (bit-exact)."""
import numpy as np
import pytest
import torch

from oracle.topk import topk_indices

pytestmark = pytest.mark.gpu


def _run(rows, k):
    import deepseek_v3_sparse_round_gb300 as dsa
    max_ctx = max(len(r) for r in rows)
    stride = dsa.dsa_score_row_stride(max_ctx)
    s = np.full((len(rows), stride), np.nan, dtype=np.float32)
    for i, r in enumerate(rows):
        s[i, :len(r)] = r
    pos = torch.tensor([len(r) - 1 for r in rows], dtype=torch.int32, device="cuda")
    out = torch.full((len(rows), k), -9, dtype=torch.int32, device="cuda")
    dsa.dsa_topk_select(torch.as_tensor(s).cuda(), pos, k, max_ctx, out)
    return out.cpu().numpy()


@pytest.mark.parametrize("k", [1, 7, 32, 2048])
def test_integer_rows_with_ties(k):
    rng = np.random.default_rng(k)
    lengths = [1, 2, k, k + 1, 3 * k + 5, 4096, 4097, 9000]
    rows = [rng.integers(-5, 6, L).astype(np.float32) for L in lengths]
    got = _run(rows, k)
    for i, r in enumerate(rows):
        assert np.array_equal(got[i], topk_indices(r, k)), (k, len(r))


@pytest.mark.parametrize("L", [40960, 40961, 65536])
def test_long_rows_shared_and_global_paths(L):
    rng = np.random.default_rng(L)
    rows = [rng.integers(-1000, 1000, L).astype(np.float32),
            np.round(rng.normal(size=L), 2).astype(np.float32)]
    got = _run(rows, 2048)
    for i, r in enumerate(rows):
        assert np.array_equal(got[i], topk_indices(r, 2048))


@pytest.mark.parametrize("L", [16383, 16384, 16385, 20003])
def test_rows_around_the_short_and_long_row_kernels(L):
    """Row lengths on both sides of the switch between the short-row and long-row kernels, with
    ragged tails (L not a multiple of 4 or of the 512-thread segment count) and heavy ties."""
    rng = np.random.default_rng(L)
    rows = [rng.integers(-20, 21, L).astype(np.float32), rng.normal(size=L).astype(np.float32),
            np.full(L, -1.25, np.float32), rng.normal(size=L - 2049).astype(np.float32)]
    for k in (2048, 1):
        got = _run(rows, k)
        for i, r in enumerate(rows):
            assert np.array_equal(got[i], topk_indices(r, k)), (L, i, k)


def test_signed_zero_and_constant_rows():
    z = np.array([-0.0, 0.0] * 50, dtype=np.float32)
    neg = -np.abs(np.random.default_rng(1).normal(size=300)).astype(np.float32)
    neg[::7] = -0.0
    rows = [z, np.full(5000, 3.5, np.float32), neg, np.zeros(3000, np.float32)]
    for k in (1, 10, 64):
        got = _run(rows, k)
        for i, r in enumerate(rows):
            assert np.array_equal(got[i], topk_indices(r, k)), (i, k)


def test_real_valued_rows_match_exactly():
    rng = np.random.default_rng(9)
    rows = [rng.normal(size=L).astype(np.float32) for L in (100, 2049, 8000, 32768)]
    got = _run(rows, 2048)
    for i, r in enumerate(rows):
        assert np.array_equal(got[i], topk_indices(r, 2048))


@pytest.mark.parametrize("k", [1, 7, 2048])
def test_batches_of_rows_of_at_most_4096(k):
    """Every row at most 4,096 long: the 256-thread kernel. Ragged lengths (not multiples of 4
    or of the thread count), heavy ties, constant and signed-zero rows, and a full 4,096 row."""
    rng = np.random.default_rng(100 + k)
    lengths = [1, 2, k, k + 1, 1000, 2049, 4093, 4095, 4096]
    rows = [rng.integers(-5, 6, L).astype(np.float32) for L in lengths]
    rows += [rng.normal(size=4096).astype(np.float32), np.full(3001, 3.5, np.float32),
             np.array([-0.0, 0.0] * 1500, dtype=np.float32)]
    got = _run(rows, k)
    for i, r in enumerate(rows):
        assert np.array_equal(got[i], topk_indices(r, k)), (k, len(r))


@pytest.mark.parametrize("L", [3000, 9000, 50000])
def test_bin_holding_exactly_the_remaining_entries(L):
    """Rows whose first radix bin (or first two) already holds exactly the entries still to
    take, so the passes stop early and every key at or above that bin is selected: k entries of
    one value above the rest, a second set where 2048 - 7 keys sit above one bin of 7, and the
    same values with one extra entry in the boundary bin (no early stop)."""
    rng = np.random.default_rng(L)
    k = 2048
    a = np.full(L, 1.0, np.float32)
    a[rng.choice(L, k, replace=False)] = 3.0                     # bin of 3.0 holds exactly k
    b = np.full(L, 0.5, np.float32)
    idx = rng.choice(L, k, replace=False)
    b[idx[:k - 7]] = 6.0
    b[idx[k - 7:]] = 2.0                                         # 7 entries in the bin of 2.0
    c = b.copy()
    c[np.flatnonzero(c == 0.5)[0]] = 2.0                         # 8 there: a tie to break
    got = _run([a, b, c], k)
    for i, r in enumerate((a, b, c)):
        assert np.array_equal(got[i], topk_indices(r, k)), (L, i)


@pytest.mark.parametrize("k", [100, 2048, 4096])
@pytest.mark.parametrize("L", [3000, 9000, 50000])
def test_output_rows_that_allow_no_wide_stores(k, L):
    """The selected indices are ranked in shared memory and stored 16 bytes at a time only when
    k <= 2048, k % 4 == 0 and the row is 16-byte aligned; an output buffer at a 4-byte offset
    (every row misaligned) and k = 4096 (too many to stage) take the direct stores: same result
    on the short-row, shared-memory and global paths, short rows' fills included."""
    import deepseek_v3_sparse_round_gb300 as dsa
    rng = np.random.default_rng(k + L)
    rows = [rng.integers(-50, 51, L).astype(np.float32), rng.normal(size=L).astype(np.float32),
            rng.normal(size=max(k - 3, 1)).astype(np.float32)]
    max_ctx = max(len(r) for r in rows)
    stride = dsa.dsa_score_row_stride(max_ctx)
    s = np.full((len(rows), stride), np.nan, dtype=np.float32)
    for i, r in enumerate(rows):
        s[i, :len(r)] = r
    pos = torch.tensor([len(r) - 1 for r in rows], dtype=torch.int32, device="cuda")
    flat = torch.full((len(rows) * k + 1,), -9, dtype=torch.int32, device="cuda")
    out = flat[1:].view(len(rows), k)                # data pointer 4 bytes past an aligned one
    assert out.data_ptr() % 16 == 4
    dsa.dsa_topk_select(torch.as_tensor(s).cuda(), pos, k, max_ctx, out)
    got = out.cpu().numpy()
    assert int(flat[0]) == -9                        # nothing written before the rows
    for i, r in enumerate(rows):
        assert np.array_equal(got[i], topk_indices(r, k)), (k, L, i)
    assert np.array_equal(_run(rows, k), got)        # the aligned buffer gives the same rows
