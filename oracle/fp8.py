"""Oracle: FP8 (E4M3) quantisation of indexer rows, and the indexer on quantised rows.

Test infrastructure only (see the package docstring).

"[DeepSeek v3.2] 上下文并行详解", section 1: the round-robin split is what allows an FP8 KV
cache. The page names no format, so the following reading is taken (stated once here and in the
design notes):

  * E4M3 as defined by the OCP 8-bit floating point format: 1 sign bit, 4 exponent bits with
    bias 7, 3 mantissa bits; subnormals at exponent field 0 (value m/8 * 2^-6); the code
    S.1111.111 is NaN, so the largest finite magnitude is 448 (S.1111.110). Rounding is to
    nearest, ties to even; magnitudes beyond 448 saturate to 448.
  * One fp32 scale per row of 128 values (one row of k_idx per token; one row of q_idx per
    (query, head)): scale = amax / 448 in fp32 (IEEE division), codes = E4M3(x / scale) with
    x / scale an IEEE fp32 division; a row of zeros gets scale 1 and zero codes. The value a code
    stands for is code * scale.
  * The indexer on quantised rows is the indexer of the dequantised values:
        I[t, s] = sum_h w[t, h] * ReLU( (sq[t, h] q8[t, h]) . (sk[s] k8[s]) )
    which, the scales being positive, equals sk[s] * sum_h (w[t, h] sq[t, h]) ReLU(q8 . k8).
  * The latent (MLA) cache in FP8, the same rule per block of 128 values: a token's 576-value
    latent row is its 512 latent values, quantised as four blocks of 128 (one fp32 scale each),
    followed by its 64 rope values kept in bf16 (the positional part the page says nothing
    about). Packed row of 656 bytes: the 512 codes, the 4 scales, the 64 bf16 rope values. The
    attention consumes bf16 rows: each latent value is bf16(fl32(code * scale)) -- the product
    rounded to fp32, then to bf16 (round to nearest, ties to even, both times); the rope values
    are the stored bf16 values.
"""
from __future__ import annotations

import numpy as np

from .indexer import indexer_scores

E4M3_MAX = 448.0
E4M3_MIN_NORMAL_EXP = -6      # 2^-6: smallest normal magnitude
E4M3_MANT_BITS = 3


def e4m3_decode(code: int) -> float:
    """Value of an 8-bit E4M3 code from its fields (NaN for S.1111.111)."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** (1 - 7)
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def e4m3_round(x) -> np.ndarray:
    """Nearest E4M3 value of each x (ties to even mantissa), saturating at +-448; fp64 out."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    out = np.zeros_like(a)
    nz = a > 0
    e = np.floor(np.log2(np.where(nz, a, 1.0)))
    e = np.maximum(e, E4M3_MIN_NORMAL_EXP)              # below 2^-6: the subnormal spacing
    quantum = np.exp2(e - E4M3_MANT_BITS)                  # spacing of the binade (exact)
    out = np.where(nz, np.rint(a / quantum) * quantum, 0.0)   # np.rint: ties to even
    out = np.minimum(out, E4M3_MAX)
    return np.copysign(out, x)


def e4m3_encode(v) -> np.ndarray:
    """Code of each value that is exactly representable in E4M3 (the output of e4m3_round)."""
    v = np.asarray(v, dtype=np.float64)
    table = {e4m3_decode(c): c for c in range(256) if not np.isnan(e4m3_decode(c))}
    table[0.0] = 0x00                                      # +0 (the rounding never makes -0 codes
    out = np.empty(v.shape, dtype=np.uint8)                # distinct: both zeros decode to 0)
    for i, val in enumerate(v.reshape(-1)):
        out.reshape(-1)[i] = table[float(val)] if val != 0 else (0x80 if np.signbit(val) else 0)
    return out


def quantize_rows(x) -> tuple:
    """Per-row FP8 quantisation: (codes' values as fp64 [rows, cols], scales fp32 [rows]).

    x: [rows, cols] (bf16 values widened). scale = fl32(amax / 448) (1 for a zero row);
    value = E4M3(fl32(x / scale))."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x32), axis=1)
    scale = np.where(amax > 0, (amax / np.float32(E4M3_MAX)).astype(np.float32),
                     np.float32(1.0)).astype(np.float32)
    ratio = (x32 / scale[:, None]).astype(np.float32)      # IEEE fp32 division
    return e4m3_round(ratio), scale


def dequantize(q_values, scales) -> np.ndarray:
    """The value each code stands for: code * scale (exact in fp64)."""
    return np.asarray(q_values, np.float64) * np.asarray(scales, np.float64)[..., None]


def indexer_scores_fp8(q8, q_scale, w, k8, k_scale, kv, pos, bid) -> list:
    """Indexer scores on FP8 rows. q8 [n_q, Hi, Di] and k8 [n_rows, Di] are E4M3 values (fp64),
    q_scale [n_q, Hi], k_scale [n_rows]: the plain indexer of the dequantised tensors."""
    q = np.asarray(q8, np.float64) * np.asarray(q_scale, np.float64)[..., None]
    k = np.asarray(k8, np.float64) * np.asarray(k_scale, np.float64)[:, None]
    return indexer_scores(q, w, k, kv, pos, bid)


# ---------------------------------------------------------------- FP8 latent (MLA) cache rows
LATENT_NOPE, LATENT_ROPE, LATENT_BLOCK = 512, 64, 128


def quantize_latent_rows(c) -> tuple:
    """Latent rows [n, 576] (bf16 values widened) -> (code values fp64 [n, 512], scales fp32
    [n, 4], rope fp64 [n, 64]): each block of 128 latent values quantised like an indexer row."""
    c = np.asarray(c, dtype=np.float64)
    n = c.shape[0]
    blocks = c[:, :LATENT_NOPE].reshape(n * (LATENT_NOPE // LATENT_BLOCK), LATENT_BLOCK)
    vals, scales = quantize_rows(blocks)
    return (vals.reshape(n, LATENT_NOPE), scales.reshape(n, LATENT_NOPE // LATENT_BLOCK),
            c[:, LATENT_NOPE:].copy())


def round_fp32_to_bf16(x) -> np.ndarray:
    """Nearest bf16 value of each fp32 value (ties to the even 8-bit significand), as fp64;
    finite inputs."""
    x32 = np.asarray(x, dtype=np.float32)
    a = np.abs(x32).astype(np.float64)
    out = np.zeros(x32.shape, dtype=np.float64)
    nz = a > 0
    e = np.floor(np.log2(np.where(nz, a, 1.0)))
    e = np.maximum(e, -126)                                 # below 2^-126: the subnormal spacing
    quantum = np.exp2(e - 7)                                # bf16 keeps 8 significant bits
    out = np.where(nz, np.rint(a / quantum) * quantum, 0.0)  # np.rint: ties to even
    return np.copysign(out, x32.astype(np.float64))


def dequantize_latent_rows(vals, scales, rope) -> np.ndarray:
    """The bf16 rows the attention reads: [n, 576] fp64 values (exactly bf16)."""
    vals = np.asarray(vals, dtype=np.float64)
    n = vals.shape[0]
    per = np.repeat(np.asarray(scales, dtype=np.float32), LATENT_BLOCK, axis=1)
    prod32 = (vals.astype(np.float32) * per).astype(np.float32)   # IEEE fp32 product
    nope = round_fp32_to_bf16(prod32)
    return np.concatenate([nope, np.asarray(rope, np.float64).reshape(n, LATENT_ROPE)], axis=1)
