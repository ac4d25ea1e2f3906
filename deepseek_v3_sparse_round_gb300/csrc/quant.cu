// FP8 (E4M3) quantisation of indexer rows (one fp32 scale per row of 128 values) and of latent
// (MLA) cache rows (the same per block of 128 latent values), and the latent rows' expansion
// back to the bf16 rows the attention reads.
//
// "[DeepSeek v3.2] 上下文并行详解", section 1: the round-robin split is what allows an FP8 KV
// cache. The page gives no format; the reading used here is E4M3 (1 sign, 4 exponent bits with
// bias 7, 3 mantissa bits, largest finite 448) with one scale per row: scale = amax / 448 and
// code = E4M3(x / scale), rounded to nearest even and saturated at +-448; a row of zeros gets
// scale 1. One warp per row: each lane holds 4 of the 128 values, a warp maximum gives amax,
// the divisions are IEEE fp32 divisions and the conversion is the hardware's round-to-nearest
// satfinite E4M3 conversion; the 128 codes of a row leave as one 128-byte store.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "status.cuh"

namespace dsa {
namespace {

constexpr int kCols = 128;
constexpr int kWarpsPerCta = 8;

__global__ void __launch_bounds__(kWarpsPerCta * 32)
quantize_rows_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows, uint8_t* __restrict__ codes,
                     float* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarpsPerCta;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5); r < rows;
       r += stride) {
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(x + r * kCols) + lane);
    const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
    const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
    const float v[4] = {__low2float(p0), __high2float(p0), __low2float(p1), __high2float(p1)};
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
        make_float2(__fdiv_rn(v[0], scale), __fdiv_rn(v[1], scale)), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
        make_float2(__fdiv_rn(v[2], scale), __fdiv_rn(v[3], scale)), __NV_SATFINITE, __NV_E4M3);
    reinterpret_cast<uint32_t*>(codes + r * kCols)[lane] =
        static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
    if (lane == 0) scales[r] = scale;
  }
}

// FP8 latent (MLA) cache rows. A token's 576-value latent row is its 512 latent values, as four
// blocks of 128 quantised like an indexer row (one fp32 scale each), then its 64 rope values,
// kept in bf16. Packed row of 656 bytes: codes [0, 512), scales [512, 528), rope [528, 656).
// The attention reads bf16 rows: a latent value expands to bf16(fl32(code * scale)), the rope
// values are copied back.
constexpr int kLatNope = 512, kLatRope = 64, kLatRow = kLatNope + kLatRope;
constexpr int kLatScales = kLatNope, kLatRopeOff = kLatNope + 4 * 4, kLatPacked = kLatRopeOff + 2 * kLatRope;
static_assert(kLatPacked == 656 && kLatPacked % 16 == 0 && kLatRopeOff % 16 == 0, "packed row");

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// One warp per row; lane l holds latent values 16l .. 16l + 15 (block l / 8).
__global__ void __launch_bounds__(kWarpsPerCta * 32)
quantize_latent_kernel(const __nv_bfloat16* __restrict__ c, int64_t rows,
                       uint8_t* __restrict__ packed) {
  const int lane = threadIdx.x & 31;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarpsPerCta;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5); r < rows;
       r += stride) {
    const uint4* src = reinterpret_cast<const uint4*>(c + r * kLatRow);
    uint8_t* dst = packed + r * kLatPacked;
    const uint4 a = __ldg(src + 2 * lane), b = __ldg(src + 2 * lane + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float v[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) { v[2 * i] = bf16_lo(w[i]); v[2 * i + 1] = bf16_hi(w[i]); }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    uint32_t q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
          make_float2(__fdiv_rn(v[4 * i], scale), __fdiv_rn(v[4 * i + 1], scale)), __NV_SATFINITE,
          __NV_E4M3);
      const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
          make_float2(__fdiv_rn(v[4 * i + 2], scale), __fdiv_rn(v[4 * i + 3], scale)),
          __NV_SATFINITE, __NV_E4M3);
      q[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
    }
    reinterpret_cast<uint4*>(dst)[lane] = make_uint4(q[0], q[1], q[2], q[3]);
    if ((lane & 7) == 0) reinterpret_cast<float*>(dst + kLatScales)[lane >> 3] = scale;
    if (lane < 8)                                    // the rope values, 16 bytes a lane
      reinterpret_cast<uint4*>(dst + kLatRopeOff)[lane] =
          __ldg(reinterpret_cast<const uint4*>(c + r * kLatRow + kLatNope) + lane);
  }
}

__global__ void __launch_bounds__(kWarpsPerCta * 32)
dequantize_latent_kernel(const uint8_t* __restrict__ packed, int64_t rows,
                         __nv_bfloat16* __restrict__ c) {
  const int lane = threadIdx.x & 31;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarpsPerCta;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5); r < rows;
       r += stride) {
    const uint8_t* src = packed + r * kLatPacked;
    uint4* dst = reinterpret_cast<uint4*>(c + r * kLatRow);
    const uint4 cw = __ldg(reinterpret_cast<const uint4*>(src) + lane);
    const float scale = __ldg(reinterpret_cast<const float*>(src + kLatScales) + (lane >> 3));
    const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
    uint32_t out[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      // two codes -> two halves (E4M3 values are exact in fp16) -> fp32 products -> bf16 pair
      const __nv_fp8x2_storage_t pair =
          static_cast<__nv_fp8x2_storage_t>((words[i >> 1] >> (16 * (i & 1))) & 0xFFFFu);
      const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
      const __nv_bfloat162 bb = __floats2bfloat162_rn(__fmul_rn(f.x, scale), __fmul_rn(f.y, scale));
      out[i] = *reinterpret_cast<const uint32_t*>(&bb);
    }
    dst[2 * lane] = make_uint4(out[0], out[1], out[2], out[3]);
    dst[2 * lane + 1] = make_uint4(out[4], out[5], out[6], out[7]);
    if (lane < 8)
      reinterpret_cast<uint4*>(c + r * kLatRow + kLatNope)[lane] =
          __ldg(reinterpret_cast<const uint4*>(src + kLatRopeOff) + lane);
  }
}

}  // namespace

int num_sms_cached();

static int latent_grid(int64_t rows) {
  const int64_t want = (rows + kWarpsPerCta - 1) / kWarpsPerCta;
  const int64_t cap = static_cast<int64_t>(num_sms_cached()) * 8;
  return static_cast<int>(want < cap ? want : cap);
}

int quantize_fp8_latent(const void* c, int64_t rows, void* packed, cudaStream_t stream) {
  if (rows < 0) return fail(DSA_ERR_INVALID, "latent quantize: rows < 0");
  if (rows == 0) return DSA_OK;
  if (!c || !packed) return fail(DSA_ERR_INVALID, "latent quantize: null pointer");
  if (reinterpret_cast<uintptr_t>(c) % 16 || reinterpret_cast<uintptr_t>(packed) % 16)
    return fail(DSA_ERR_INVALID, "latent quantize: rows must be 16-byte aligned");
  quantize_latent_kernel<<<latent_grid(rows), kWarpsPerCta * 32, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(c), rows, static_cast<uint8_t*>(packed));
  DSA_CHECK_CUDA(cudaGetLastError());
  return DSA_OK;
}

int dequantize_fp8_latent(const void* packed, int64_t rows, void* c, cudaStream_t stream) {
  if (rows < 0) return fail(DSA_ERR_INVALID, "latent dequantize: rows < 0");
  if (rows == 0) return DSA_OK;
  if (!c || !packed) return fail(DSA_ERR_INVALID, "latent dequantize: null pointer");
  if (reinterpret_cast<uintptr_t>(c) % 16 || reinterpret_cast<uintptr_t>(packed) % 16)
    return fail(DSA_ERR_INVALID, "latent dequantize: rows must be 16-byte aligned");
  dequantize_latent_kernel<<<latent_grid(rows), kWarpsPerCta * 32, 0, stream>>>(
      static_cast<const uint8_t*>(packed), rows, static_cast<__nv_bfloat16*>(c));
  DSA_CHECK_CUDA(cudaGetLastError());
  return DSA_OK;
}

int quantize_fp8_rows(const void* x, int64_t rows, int cols, void* codes, float* scales,
                      cudaStream_t stream) {
  if (rows < 0) return fail(DSA_ERR_INVALID, "quantize: rows < 0");
  if (cols != kCols)
    return fail(DSA_ERR_UNSUPPORTED, "quantize: rows of %d values not built; supported 128", cols);
  if (rows == 0) return DSA_OK;
  if (!x || !codes || !scales) return fail(DSA_ERR_INVALID, "quantize: null pointer");
  if (reinterpret_cast<uintptr_t>(x) % 8 || reinterpret_cast<uintptr_t>(codes) % 4 ||
      reinterpret_cast<uintptr_t>(scales) % 4)
    return fail(DSA_ERR_INVALID, "quantize: x must be 8-byte and codes 4-byte aligned");
  const int64_t want = (rows + kWarpsPerCta - 1) / kWarpsPerCta;
  const int64_t cap = static_cast<int64_t>(num_sms_cached()) * 8;
  const int grid = static_cast<int>(want < cap ? want : cap);
  quantize_rows_kernel<<<grid, kWarpsPerCta * 32, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(x), rows, static_cast<uint8_t*>(codes), scales);
  DSA_CHECK_CUDA(cudaGetLastError());
  return DSA_OK;
}

}  // namespace dsa
