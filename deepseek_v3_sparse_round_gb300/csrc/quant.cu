// FP8 (E4M3) quantisation of indexer rows: one fp32 scale per row of 128 values.
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

}  // namespace

int num_sms_cached();

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
