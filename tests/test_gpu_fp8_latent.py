"""GPU parity for the FP8 latent (MLA) cache rows: packing bit for bit against the oracle (codes,
block scales, rope bytes), the expansion to bf16 bit for bit (from the kernel's own packing and
from arbitrary codes and scales), and the sparse MLA on a cache that went through FP8 -- packed,
split and all-gathered as 656-byte rows, reranged, expanded -- against the oracle's MLA on the
oracle's expanded rows."""
import numpy as np
import pytest
import torch

import workloads as W
from dsa_cases import Shard, f64, i32, mla_close
from oracle import fp8 as ofp8
from oracle import mla as omla

pytestmark = pytest.mark.gpu


def _dsa():
    import deepseek_v3_sparse_round_gb300 as dsa
    return dsa


def _rows(n, seed):
    """bf16 latent rows with per-row magnitudes from 2^-20 to 2^20, a zero block, a block with
    one large entry, and subnormal-scaled blocks."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.randn(n, 576, generator=g) * torch.exp2(torch.randint(-20, 21, (n, 1), generator=g).float())
    if n > 3:
        x[1, 128:256] = 0.0
        x[2, 300] = 3.0e4
        x[3, :512] *= 2.0 ** -100
    return x.to(torch.bfloat16).cuda()


def _unpack(packed):
    p = packed.cpu().numpy()
    codes = p[:, :512]
    scales = p[:, 512:528].copy().view(np.float32)
    rope = torch.from_numpy(p[:, 528:656].copy()).view(torch.bfloat16).float().numpy().astype(np.float64)
    return codes, scales, rope


@pytest.mark.parametrize("n", [1, 7, 4096, 70001])
def test_packing_matches_the_oracle_bit_for_bit(n):
    dsa = _dsa()
    c = _rows(n, n)
    packed = torch.full((n, 656), 0xEE, dtype=torch.uint8, device="cuda")
    dsa.dsa_quantize_fp8_latent(c, packed)
    codes, scales, rope = _unpack(packed)
    vals, s_ref, rope_ref = ofp8.quantize_latent_rows(f64(c))
    assert np.array_equal(scales, s_ref)
    assert np.array_equal(codes, ofp8.e4m3_encode(vals).reshape(codes.shape))
    assert np.array_equal(rope, rope_ref)
    # the expansion of the packed rows: bit for bit the oracle's bf16 rows
    back = torch.empty_like(c)
    dsa.dsa_dequantize_fp8_latent(packed, back)
    assert np.array_equal(f64(back), ofp8.dequantize_latent_rows(vals, s_ref, rope_ref))


def test_expansion_of_arbitrary_codes_and_scales():
    dsa = _dsa()
    rng = np.random.default_rng(5)
    n = 3000
    finite = np.array([cde for cde in range(256) if cde not in (0x7F, 0xFF)], dtype=np.uint8)
    codes = rng.choice(finite, size=(n, 512)).astype(np.uint8)
    scales = (rng.uniform(0.5, 2.0, (n, 4)) * 2.0 ** rng.integers(-130, 100, (n, 4))).astype(np.float32)
    scales[0, 0] = np.float32(2.0 ** -149)               # products down in the subnormal range
    rope = torch.randn(n, 64, dtype=torch.float32).to(torch.bfloat16)
    packed = np.concatenate([codes, scales.view(np.uint8).reshape(n, 16),
                             rope.view(torch.uint8).numpy().reshape(n, 128)], axis=1)
    p_dev = torch.from_numpy(packed).cuda()
    out = torch.empty((n, 576), dtype=torch.bfloat16, device="cuda")
    dsa.dsa_dequantize_fp8_latent(p_dev, out)
    vals = np.vectorize(ofp8.e4m3_decode)(codes.astype(np.int64))
    ref = ofp8.dequantize_latent_rows(vals, scales, rope.float().numpy().astype(np.float64))
    assert np.array_equal(f64(out), ref)


def test_rejects_bad_arguments():
    dsa = _dsa()
    c = torch.zeros((4, 576), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        dsa.dsa_quantize_fp8_latent(c, torch.zeros((4, 655), dtype=torch.uint8, device="cuda"))
    with pytest.raises(ValueError):
        dsa.dsa_dequantize_fp8_latent(torch.zeros((4, 656), dtype=torch.uint8, device="cuda"),
                                      torch.zeros((4, 512), dtype=torch.bfloat16, device="cuda"))
    flat = torch.zeros(4 * 656 + 8, dtype=torch.uint8, device="cuda")
    with pytest.raises(RuntimeError):                    # packed rows not 16-byte aligned
        dsa.dsa_quantize_fp8_latent(c, flat[8:].view(4, 656))
    dsa.dsa_quantize_fp8_latent(c[:0], flat[:0].view(0, 656))   # no rows: nothing to do


@pytest.mark.parametrize("wid,rank", [(1, 3), (3, 1)])
def test_sparse_mla_on_a_cache_that_went_through_fp8(wid, rank):
    """Logical latent rows -> FP8 packed rows -> each rank's split gathers its packed rows ->
    the all-gathered packed rows are reranged -> expanded to bf16 -> sparse MLA, against the
    oracle's MLA over the oracle's expanded rows (top-k sets from the oracle)."""
    dsa = _dsa()
    sh = Shard(W.WORKLOADS[wid], rank, integer_indexer=False)
    wl, N = sh.wl, sh.n_rows
    c = sh.mla.c.cuda()
    packed = torch.empty((N, 656), dtype=torch.uint8, device="cuda")
    dsa.dsa_quantize_fp8_latent(c, packed)
    gathered = []
    for r in range(wl.sp):
        m = dsa.dsa_rr_shard_len(N, wl.sp, r)
        cs = torch.empty(sh.n_req + 1, dtype=torch.int32, device="cuda")
        p, b, g = (torch.empty(m, dtype=torch.int32, device="cuda") for _ in range(3))
        dst = torch.empty((m, 656), dtype=torch.uint8, device="cuda")
        dsa.dsa_rr_split_metadata(sh.d_cu, N, wl.sp, r, cs, p, b, g, src_rows=packed, dst_rows=dst)
        gathered.append(dst)
    logical = torch.empty_like(packed)
    dsa.dsa_rr_rerange(torch.cat(gathered), logical, N, wl.sp, 0)
    assert torch.equal(logical, packed)
    c8 = torch.empty_like(c)
    dsa.dsa_dequantize_fp8_latent(logical, c8)
    sel = sh.samples(24)
    view = sh.oracle_view(sel)
    topk_np = sh.oracle_topk(sh.oracle_scores(sel, view))
    sel_t = torch.as_tensor(sel, device="cuda")
    o = torch.empty((len(sel), wl.H, wl.dv), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((len(sel), wl.H), dtype=torch.float32, device="cuda")
    dsa.dsa_sparse_mla(sh.mla.q[sel_t].cuda(), c8, sh.d_cu, sh.n_req, i32(sh.bid[sel]),
                       i32(topk_np), wl.scale, o, lse)
    torch.cuda.synchronize()
    assert dsa.dsa_read_device_errors() == 0
    vals, scales, rope = ofp8.quantize_latent_rows(f64(c))
    c_exp = ofp8.dequantize_latent_rows(vals, scales, rope)
    ref_o, ref_lse = omla.sparse_mla(view["q"], c_exp[view["row_ids"]], view["kv"], view["bid"],
                                     topk_np, wl.scale, wl.dv)
    mla_close(f64(o), ref_o)
    assert np.allclose(lse.cpu().numpy(), ref_lse, atol=1e-3, rtol=1e-4)
