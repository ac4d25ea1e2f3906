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
@pytest.mark.parametrize("width", [576, 128])          # latent rows (1152 B), k_idx rows (256 B)
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
