"""GPU: the row-gather rate probe runs every mechanism (cp.async, TMA tile::gather4, registers,
DSMEM, TMA boxes of consecutive rows) to completion on a small case, with every CTA reporting its cycle count and no device error; rows
outside the cache are reported, not read."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def _case(n_rows=1000, n_ctas=4, n_tiles=7, seed=0):
    g = torch.Generator(device="cpu").manual_seed(seed)
    c = torch.randn(n_rows, 576, generator=g).to(torch.bfloat16).cuda()
    rows = torch.randint(0, n_rows, (n_ctas * n_tiles * 48,), generator=g, dtype=torch.int32).cuda()
    return c, rows, torch.zeros(n_ctas, dtype=torch.int64, device="cuda")


@pytest.mark.parametrize("mode,issuers", [(0, 1), (1, 1), (1, 5), (1, 32), (2, 1), (3, 1), (4, 1), (5, 1), (6, 1), (7, 1)])
def test_probe_runs_clean(mode, issuers):
    import deepseek_v3_sparse_round_gb300 as dsa
    dsa.dsa_read_device_errors()
    c, rows, cycles = _case()
    dsa.dsa_probe_row_gather(c, rows, 4, 7, mode, issuers, cycles)
    torch.cuda.synchronize()
    assert dsa.dsa_read_device_errors() == 0
    assert bool((cycles > 0).all())


def test_probe_flags_rows_outside_the_cache():
    import deepseek_v3_sparse_round_gb300 as dsa
    dsa.dsa_read_device_errors()
    c, rows, cycles = _case()
    rows[5] = 1000                                   # n_rows: one past the end
    rows[77] = -3
    dsa.dsa_probe_row_gather(c, rows, 4, 7, 0, 1, cycles)
    assert dsa.dsa_read_device_errors() & dsa.DEVERR_BAD_INDEX


def test_probe_rejects_bad_arguments():
    import deepseek_v3_sparse_round_gb300 as dsa
    c, rows, cycles = _case()
    with pytest.raises(ValueError):
        dsa.dsa_probe_row_gather(c, rows[:-1], 4, 7, 0, 1, cycles)
    with pytest.raises(RuntimeError):
        dsa.dsa_probe_row_gather(c, rows, 4, 7, 8, 1, cycles)
    with pytest.raises(RuntimeError):
        dsa.dsa_probe_row_gather(c, rows, 4, 7, 1, 33, cycles)
