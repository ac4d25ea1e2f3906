"""GPU parity for the FP8 (E4M3) indexer rows: the quantisation kernel bit for bit against the
oracle's rounding, and the tensor-core FP8 indexer + top-k against the oracle's indexer of the
dequantised rows (exact on integer codes with power-of-two scales; within a derived bound on
bf16 N(0,1) rows quantised by the kernel)."""
import numpy as np
import pytest
import torch

import workloads as W
from dsa_cases import Shard, check_topk_near_ties, dsa, f64, i32
from oracle import fp8 as ofp8
from oracle.kv import ContiguousKV

pytestmark = pytest.mark.gpu

_DECODE = np.array([ofp8.e4m3_decode(c) for c in range(256)])


def _values(codes: torch.Tensor) -> np.ndarray:
    return _DECODE[codes.cpu().numpy().astype(np.int64)]


@pytest.mark.parametrize("rows", [1, 7, 4096, 70001])
def test_quantize_rows_bit_exact(rows):
    m = dsa()
    x = W.normal_bf16((rows, 128), seed=rows, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(3)
    x = (x.float() * torch.exp2(torch.randint(-12, 12, (rows, 1), generator=g, device="cuda")
                                .float())).to(torch.bfloat16)
    if rows > 7:
        x[3] = 0                                         # a zero row: scale 1, zero codes
        x[5] = 0
        x[5, 77] = -1.5                                  # one non-zero entry: it maps to -448
        x[6] = x[6] * 1e-30                              # subnormal codes in the row
    codes = torch.empty((rows, 128), dtype=torch.uint8, device="cuda")
    scales = torch.empty(rows, dtype=torch.float32, device="cuda")
    m.dsa_quantize_fp8_rows(x, codes, scales)
    q_ref, s_ref = ofp8.quantize_rows(f64(x))
    assert np.array_equal(scales.cpu().numpy(), s_ref)
    got = _values(codes)
    assert np.array_equal(got, q_ref)
    # the kernel's zero codes are +0 (0x00) or -0 (0x80); both stand for 0
    assert not np.isnan(got).any()


def test_quantize_q_idx_layout():
    """q_idx [n_q, Hi, 128] quantises per (query, head) row: scales [n_q, Hi]."""
    m = dsa()
    x = W.normal_bf16((33, 64, 128), seed=9, device="cuda")
    codes = torch.empty_like(x, dtype=torch.uint8)
    scales = torch.empty((33, 64), dtype=torch.float32, device="cuda")
    m.dsa_quantize_fp8_rows(x, codes, scales)
    q_ref, s_ref = ofp8.quantize_rows(f64(x).reshape(-1, 128))
    assert np.array_equal(scales.cpu().numpy().reshape(-1), s_ref)
    assert np.array_equal(_values(codes).reshape(-1, 128), q_ref)


class Fp8Shard:
    """A shard's indexer inputs as E4M3 codes with fp32 scales."""

    def __init__(self, wid, rank, integer=True, max_ctx=None):
        self.sh = Shard(W.WORKLOADS[wid], rank, integer_indexer=False)
        sh, wl = self.sh, self.sh.wl
        if max_ctx is not None:
            sh.max_ctx = max_ctx
        if integer:
            self.q8 = W.int_codes_e4m3((sh.n_q, wl.Hi, wl.Di), -3, 3, 500 + rank, device="cuda")
            self.k8 = W.int_codes_e4m3((sh.n_rows, wl.Di), -3, 3, 501, device="cuda")
            self.qs = W.pow2_scales((sh.n_q, wl.Hi), -2, 2, 502 + rank, device="cuda")
            self.ks = W.pow2_scales((sh.n_rows,), -2, 2, 503, device="cuda")
            self.w = W.int_uniform((sh.n_q, wl.Hi), -3, 3, 504 + rank, dtype=torch.float32,
                                   device="cuda")
        else:                                            # the kernel quantises bf16 rows
            m = dsa()
            self.q8 = torch.empty((sh.n_q, wl.Hi, wl.Di), dtype=torch.uint8, device="cuda")
            self.qs = torch.empty((sh.n_q, wl.Hi), dtype=torch.float32, device="cuda")
            self.k8 = torch.empty((sh.n_rows, wl.Di), dtype=torch.uint8, device="cuda")
            self.ks = torch.empty(sh.n_rows, dtype=torch.float32, device="cuda")
            m.dsa_quantize_fp8_rows(sh.idx.q_idx.cuda(), self.q8, self.qs)
            m.dsa_quantize_fp8_rows(sh.idx.k_idx.cuda(), self.k8, self.ks)
            self.w = sh.idx.w.cuda()

    def scores(self):
        m, sh = dsa(), self.sh
        stride = m.dsa_score_row_stride(sh.max_ctx)
        out = torch.full((sh.n_q, stride), float("nan"), device="cuda")
        ws = torch.empty(m.dsa_indexer_topk_workspace_size(sh.n_q, sh.max_ctx, sh.wl.topk),
                         dtype=torch.uint8, device="cuda")
        m.dsa_indexer_scores_fp8(self.q8, self.qs, self.w, self.k8, self.ks, sh.d_cu, sh.n_req,
                                 sh.d_pos, sh.d_bid, sh.max_ctx, out, ws,
                                 block_table=sh.block_table)
        return out

    def topk(self):
        m, sh = dsa(), self.sh
        ws = torch.empty(m.dsa_indexer_topk_workspace_size(sh.n_q, sh.max_ctx, sh.wl.topk),
                         dtype=torch.uint8, device="cuda")
        out = torch.full((sh.n_q, sh.wl.topk), -9, dtype=torch.int32, device="cuda")
        m.dsa_indexer_topk_fp8(self.q8, self.qs, self.w, self.k8, self.ks, sh.d_cu, sh.n_req,
                               sh.d_pos, sh.d_bid, sh.wl.topk, sh.max_ctx, out, ws,
                               block_table=sh.block_table)
        return out

    def oracle(self, sel):
        """Oracle scores of queries `sel` on the dequantised rows (each request's keys packed
        the way Shard.oracle_view packs them)."""
        sh = self.sh
        sel = np.asarray(sel, dtype=np.int64)
        reqs = sorted(set(int(b) for b in sh.bid[sel]))
        need = {b: int(sh.pos[sel][sh.bid[sel] == b].max()) + 1 for b in reqs}
        rows = np.concatenate([sh.kv.rows(b, np.arange(need[b])) for b in reqs])
        cu2 = np.concatenate([[0], np.cumsum([need[b] for b in reqs])]).astype(np.int64)
        remap = {b: i for i, b in enumerate(reqs)}
        st = torch.as_tensor(sel, device="cuda")
        r = torch.as_tensor(rows, device="cuda")
        return ofp8.indexer_scores_fp8(_values(self.q8[st]), f64(self.qs[st]), f64(self.w[st]),
                                       _values(self.k8[r]), f64(self.ks[r]), ContiguousKV(cu2),
                                       sh.pos[sel],
                                       np.asarray([remap[int(b)] for b in sh.bid[sel]]))


@pytest.mark.parametrize("wid,rank", [(1, 3), (2, 6), (3, 0), (4, 0)])
def test_fp8_indexer_integer_codes_exact(wid, rank):
    """Integer E4M3 codes with power-of-two scales: every score is exact in fp32, so scores
    and index sets match the oracle bit for bit (and the fused path, max_ctx > 8192, equals the
    separate one)."""
    f = Fp8Shard(wid, rank, integer=True)
    sh = f.sh
    sel = sh.samples(24)
    ora = f.oracle(sel)
    s_np = f.scores().cpu().numpy()
    t_np = f.topk().cpu().numpy()
    ora_topk = sh.oracle_topk(ora)
    for i, t in enumerate(sel):
        L = int(sh.pos[t]) + 1
        assert np.array_equal(s_np[t, :L].astype(np.float64), ora[i]), (t, L)
        assert np.array_equal(t_np[t], ora_topk[i]), t
    assert dsa().dsa_read_device_errors() == 0


def test_fp8_fused_path_forced_on_short_rows():
    f = Fp8Shard(1, 3, integer=True, max_ctx=9000)
    sh = f.sh
    sel = sh.samples(32)
    ora_topk = sh.oracle_topk(f.oracle(sel))
    t_np = f.topk().cpu().numpy()
    for i, t in enumerate(sel):
        assert np.array_equal(t_np[t], ora_topk[i]), t


@pytest.mark.parametrize("wid,rank", [(1, 3), (4, 0)])
def test_fp8_indexer_bf16_rows_within_bound(wid, rank):
    """bf16 N(0,1) rows quantised by the kernel: scores within a bound of the oracle on the same
    codes and scales, index sets equal except at near-ties. Each E4M3 x E4M3 product is exact
    in fp32; the tensor core sums 128 of them per head and the epilogue sums the heads, so the
    error is at most (Di + Hi) 2^-24 of the sum of magnitudes (plus the two scale products); the
    test allows 2^-20 (Di + Hi) to leave room for the tensor core's internal accumulation."""
    f = Fp8Shard(wid, rank, integer=False)
    sh, wl = f.sh, f.sh.wl
    sel = sh.samples(24)
    ora = f.oracle(sel)
    s_np = f.scores().cpu().numpy()
    t_np = f.topk().cpu().numpy()
    st = torch.as_tensor(sel, device="cuda")
    q = _values(f.q8[st]) * f64(f.qs[st])[..., None]
    w = np.abs(f64(f.w[st]))
    for i, t in enumerate(sel):
        L = int(sh.pos[t]) + 1
        rows = sh.kv.rows(int(sh.bid[t]), np.arange(L))
        kk = np.abs(_values(f.k8[torch.as_tensor(rows, device="cuda")]) *
                    f64(f.ks[torch.as_tensor(rows, device="cuda")])[:, None])
        mag = w[i] @ (np.abs(q[i]) @ kk.T)
        err = np.abs(s_np[t, :L].astype(np.float64) - ora[i])
        assert np.all(err <= 2.0 ** -20 * (wl.Di + wl.Hi) * mag + 1e-30), t
        check_topk_near_ties(t_np[t], sh.oracle_topk([ora[i]])[0], ora[i], wl.topk)
