"""Pins for the FP8 (E4M3) oracle (no GPU): the format's fixed code points, round-to-nearest
with ties to even against brute force over every code, saturation, per-row scaling, and the
indexer on quantised rows against brute-force loops."""
import numpy as np
import pytest

from oracle import fp8
from oracle.kv import ContiguousKV


def test_code_points_of_the_format():
    # OCP 8-bit floating point specification (OFP8), E4M3: exponent bias 7, 3 mantissa bits,
    # S.1111.111 is NaN; these code points are fixed by that definition.
    assert fp8.e4m3_decode(0x7E) == 448.0                  # largest finite
    assert fp8.e4m3_decode(0x08) == 2.0 ** -6              # smallest normal
    assert fp8.e4m3_decode(0x07) == 7 * 2.0 ** -9          # largest subnormal
    assert fp8.e4m3_decode(0x01) == 2.0 ** -9              # smallest subnormal
    assert fp8.e4m3_decode(0x38) == 1.0 and fp8.e4m3_decode(0xB8) == -1.0
    assert fp8.e4m3_decode(0x3C) == 1.5 and fp8.e4m3_decode(0x40) == 2.0
    assert np.isnan(fp8.e4m3_decode(0x7F)) and np.isnan(fp8.e4m3_decode(0xFF))
    assert fp8.e4m3_decode(0x00) == 0.0


def _finite_codes():
    return [c for c in range(256) if not np.isnan(fp8.e4m3_decode(c))]


def test_every_finite_value_rounds_to_itself():
    v = np.array([fp8.e4m3_decode(c) for c in _finite_codes()])
    assert np.array_equal(fp8.e4m3_round(v), v)
    codes = fp8.e4m3_encode(v)
    assert all(fp8.e4m3_decode(int(c)) == x for c, x in zip(codes, v))


def test_ties_go_to_the_even_mantissa():
    assert fp8.e4m3_round(1.0625) == 1.0                   # between 1.0 (m=0) and 1.125 (m=1)
    assert fp8.e4m3_round(1.1875) == 1.25                  # between 1.125 (m=1) and 1.25 (m=2)
    assert fp8.e4m3_round(2.0 ** -10) == 0.0               # between 0 and 2^-9
    assert fp8.e4m3_round(3 * 2.0 ** -10) == 2.0 ** -8     # between 2^-9 (m=1) and 2^-8 (m=2)
    assert fp8.e4m3_round(-1.0625) == -1.0


def test_saturation_to_the_largest_finite():
    assert fp8.e4m3_round(448.0) == 448.0
    assert fp8.e4m3_round(463.9) == 448.0
    assert fp8.e4m3_round(500.0) == 448.0 and fp8.e4m3_round(-1e6) == -448.0


def test_rounding_is_nearest_by_brute_force():
    codes = _finite_codes()
    vals = np.array([fp8.e4m3_decode(c) for c in codes])
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(size=2000) * 10.0 ** rng.integers(-4, 3, 2000),
                        rng.uniform(-448, 448, 500), [0.0, -0.0]])
    got = fp8.e4m3_round(x)
    for xi, gi in zip(x, got):
        d = np.abs(vals - xi)
        best = np.flatnonzero(d == d.min())
        if len(best) > 1:                                  # a tie: the even mantissa wins
            best = [b for b in best if codes[b] & 1 == 0]
        assert gi == vals[best[0]] or (gi == 0 and vals[best[0]] == 0), (xi, gi)


def test_row_quantisation_scale_and_error_bound():
    rng = np.random.default_rng(1)
    x = (rng.normal(size=(64, 128)) * rng.uniform(0.01, 30, (64, 1))).astype(np.float32)
    x[3] = 0.0
    x[4] = 0.0
    x[4, 17] = -2.5
    q, s = fp8.quantize_rows(x)
    assert s.dtype == np.float32 and s[3] == 1.0 and np.all(q[3] == 0)
    am = np.argmax(np.abs(x), axis=1)
    for r in range(64):
        if r == 3:
            continue
        assert abs(q[r, am[r]]) == 448.0                   # the largest entry maps to +-448
        assert s[r] == np.float32(np.max(np.abs(x[r])) / np.float32(448.0))
    deq = fp8.dequantize(q, s)
    bound = np.maximum(2.0 ** -4 * np.abs(x), 2.0 ** -10 * s[:, None]) * (1 + 1e-6)
    assert np.all(np.abs(deq - x) <= bound)
    assert q[4, 17] == -448.0 and np.count_nonzero(q[4]) == 1


def test_indexer_on_quantised_rows_brute_force():
    rng = np.random.default_rng(2)
    Hi, Di, n = 3, 8, 12
    cu = np.array([0, 5, 12])
    k8 = rng.integers(-3, 4, (n, Di)).astype(np.float64)
    q8 = rng.integers(-3, 4, (4, Hi, Di)).astype(np.float64)
    ks = 2.0 ** rng.integers(-3, 3, n)
    qs = 2.0 ** rng.integers(-3, 3, (4, Hi))
    w = rng.integers(-2, 3, (4, Hi)).astype(np.float64)
    pos = np.array([0, 4, 2, 6])
    bid = np.array([0, 0, 1, 1])
    got = fp8.indexer_scores_fp8(q8, qs, w, k8, ks, ContiguousKV(cu), pos, bid)
    for t in range(4):
        for s_ in range(pos[t] + 1):
            row = cu[bid[t]] + s_
            want = 0.0
            for h in range(Hi):
                dot = sum(q8[t, h, d] * qs[t, h] * k8[row, d] * ks[row] for d in range(Di))
                want += w[t, h] * max(dot, 0.0)
            assert got[t][s_] == want
        # the scales factor out of the ReLU: sk * sum_h (w sq) ReLU(q8 . k8)
        for s_ in range(pos[t] + 1):
            row = cu[bid[t]] + s_
            alt = ks[row] * sum(w[t, h] * qs[t, h] * max(q8[t, h] @ k8[row], 0.0) for h in range(Hi))
            assert np.isclose(got[t][s_], alt, rtol=0, atol=1e-12)


# ------------------------------------------------ FP8 latent (MLA) cache rows
def test_bf16_rounding_against_the_library_conversion():
    import torch
    rng = np.random.default_rng(7)
    x = (rng.normal(size=20000) * 10.0 ** rng.integers(-30, 30, 20000)).astype(np.float32)
    ties = np.float32(1.0) + np.float32(2.0 ** -8) * np.arange(1, 8, 2, dtype=np.float32)  # halfway
    tiny = (np.arange(1, 200, dtype=np.float32) * np.float32(2.0 ** -140))                   # subnormal
    x = np.concatenate([x[np.isfinite(x)], ties, -ties, tiny, [0.0, -0.0]]).astype(np.float32)
    ref = torch.tensor(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(fp8.round_fp32_to_bf16(x), ref)


def test_latent_blocks_scale_rope_and_zero_block():
    rng = np.random.default_rng(3)
    c = rng.normal(size=(3, 576))
    c[1, 128:256] = 0.0                                   # a zero block: scale 1, codes 0
    c[2, 300] = -50.0                                     # block 2's largest magnitude
    vals, scales, rope = fp8.quantize_latent_rows(c)
    assert vals.shape == (3, 512) and scales.shape == (3, 4) and rope.shape == (3, 64)
    assert np.array_equal(rope, c[:, 512:])               # the rope part is not quantised
    assert scales[1, 1] == 1.0 and np.all(vals[1, 128:256] == 0.0)
    assert scales[2, 2] == np.float32(50.0 / 448.0) and vals[2, 300] == -448.0
    for r in range(3):
        for b in range(4):
            blk = c[r, 128 * b:128 * (b + 1)]
            if np.any(blk):
                assert np.max(np.abs(vals[r, 128 * b:128 * (b + 1)])) == 448.0
                assert scales[r, b] == np.float32(np.float32(np.max(np.abs(blk))) / np.float32(448))


def test_latent_dequantised_values():
    vals = np.zeros((1, 512)); scales = np.ones((1, 4), np.float32)
    vals[0, 0], scales[0, 0] = 448.0, np.float32(2.0)     # 896: exact in bf16
    vals[0, 128], scales[0, 1] = 1.0, np.float32(0.1)     # fp32 0.1, then bf16: 0.10009765625
    vals[0, 256], scales[0, 2] = 1.125, np.float32(3.0)   # 3.375 (8 significant bits suffice)
    vals[0, 384], scales[0, 3] = 1.875, np.float32(1.0 + 2.0 ** -7)   # 1.889648..., rounded
    rope = np.arange(64, dtype=np.float64).reshape(1, 64)
    out = fp8.dequantize_latent_rows(vals, scales, rope)
    assert out[0, 0] == 896.0 and out[0, 128] == 0.10009765625 and out[0, 256] == 3.375
    exact = 1.875 * (1.0 + 2.0 ** -7)                     # 1.8896484375 = 1.1110001111... in binary
    assert out[0, 384] == 1.890625 and abs(out[0, 384] - exact) <= 2.0 ** -8
    assert np.array_equal(out[0, 512:], rope[0])


def test_latent_round_trip_within_the_format_bound():
    rng = np.random.default_rng(11)
    c = rng.normal(size=(64, 576)) * 10.0 ** rng.integers(-3, 3, (64, 1))
    vals, scales, rope = fp8.quantize_latent_rows(c)
    back = fp8.dequantize_latent_rows(vals, scales, rope)
    per = np.repeat(scales.astype(np.float64), 128, axis=1)
    x = c[:, :512].astype(np.float32).astype(np.float64)
    # E4M3: half a spacing, 2^-4 relative for normal codes, 2^-10 scale in the subnormal range;
    # then the fp32 and bf16 roundings of the product
    bound = 2.0 ** -4 * np.abs(x) + 2.0 ** -10 * per + 2.0 ** -8 * np.abs(back[:, :512])
    assert np.all(np.abs(back[:, :512] - x) <= bound)
    assert np.array_equal(back[:, 512:], c[:, 512:])
