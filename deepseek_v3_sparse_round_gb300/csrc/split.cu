// Round-robin split metadata + row gather, and the rerange of an all-gathered buffer.
//
// "[DeepSeek v3.2] 上下文并行详解", section 2.B: rank r keeps the flattened tokens
// r, r+sp, r+2sp, ... and a metadata kernel recomputes cu_seqlens and batch indices after the
// scatter. Section 4 part 3 step B: the all-gathered rows arrive rank by rank and are put back
// in logical order. Both kernels are plain HBM streams: 16-byte vector loads and stores over
// the flattened (row, 16-byte chunk) index space, several independent chunks in flight per
// thread, grid sized to a multiple of the SM count.
#include <cstdint>
#include <cuda_runtime.h>

#include "status.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

__device__ __forceinline__ int4 ld_stream(const int4* p) {
  int4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void st_stream(int4* p, int4 v) {
  asm volatile("st.global.L1::no_allocate.v4.s32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Number of flattened tokens g < x with g = rank (mod sp): max(0, ceil((x - rank) / sp)).
__device__ __forceinline__ int32_t shard_count_below(int64_t x, int sp, int rank) {
  const int64_t d = x - rank;
  return d <= 0 ? 0 : static_cast<int32_t>((d + sp - 1) / sp);
}

// Largest b in [0, n_req) with cu[b] <= g (cu non-decreasing, cu[0] = 0 <= g < cu[n_req]).
__device__ __forceinline__ int find_request(const int32_t* cu, int n_req, int64_t g) {
  int lo = 0, hi = n_req - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<int64_t>(__ldg(cu + mid)) <= g) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kThreads)
split_meta_kernel(const int32_t* __restrict__ cu, int n_req, int64_t n_r, int sp, int rank,
                  int32_t* __restrict__ cu_shard, int32_t* __restrict__ pos,
                  int32_t* __restrict__ bid, int32_t* __restrict__ gidx) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (int64_t i = i0; i <= n_req; i += stride)
    cu_shard[i] = shard_count_below(__ldg(cu + i), sp, rank);
  for (int64_t t = i0; t < n_r; t += stride) {
    const int64_t g = rank + t * sp;
    const int b = find_request(cu, n_req, g);
    pos[t] = static_cast<int32_t>(g - __ldg(cu + b));
    bid[t] = b;
    if (gidx) gidx[t] = static_cast<int32_t>(g);
  }
}

// Source row of destination row `r` for the two copy patterns.
struct SplitRows {
  int sp, rank;
  __device__ __forceinline__ int64_t operator()(int64_t t) const { return rank + t * sp; }
};
struct RerangeRows {
  int sp;
  int64_t per_rank;   // floor(N / sp) (packed) -- unused when padded
  int64_t rem;        // N % sp (packed)
  int64_t stride;     // > 0: padded blocks
  __device__ __forceinline__ int64_t operator()(int64_t g) const {
    const int64_t q = g % sp, j = g / sp;
    const int64_t off = stride > 0 ? q * stride : q * per_rank + (q < rem ? q : rem);
    return off + j;
  }
};

template <class RowMap>
__global__ void __launch_bounds__(kThreads)
copy_rows_v16_kernel(const int4* __restrict__ src, int4* __restrict__ dst, int64_t n_rows,
                     int64_t chunks_per_row, RowMap map) {
  const int64_t total = n_rows * chunks_per_row;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + (kUnroll - 1) * stride < total; i += kUnroll * stride) {
    int4 v[kUnroll];
    int64_t di[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t c = i + u * stride;
      const int64_t r = c / chunks_per_row, col = c - r * chunks_per_row;
      di[u] = c;
      v[u] = ld_stream(src + map(r) * chunks_per_row + col);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) st_stream(dst + di[u], v[u]);
  }
  for (; i < total; i += stride) {
    const int64_t r = i / chunks_per_row, col = i - r * chunks_per_row;
    st_stream(dst + i, ld_stream(src + map(r) * chunks_per_row + col));
  }
}

template <class RowMap>
__global__ void __launch_bounds__(kThreads)
copy_rows_bytes_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                       int64_t n_rows, int64_t row_bytes, RowMap map) {
  const int64_t total = n_rows * row_bytes;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int64_t r = i / row_bytes, col = i - r * row_bytes;
    dst[i] = src[map(r) * row_bytes + col];
  }
}

int num_sms() {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0)
      sms = 148;
  }
  return sms;
}

int grid_for(int64_t work_items, int per_thread) {
  const int64_t want = (work_items + static_cast<int64_t>(kThreads) * per_thread - 1) /
                       (static_cast<int64_t>(kThreads) * per_thread);
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;   // 8 x 256-thread CTAs per SM
  int64_t g = want < cap ? want : cap;
  return g < 1 ? 1 : static_cast<int>(g);
}

template <class RowMap>
int launch_copy_rows(const void* src, void* dst, int64_t n_rows, int64_t row_bytes, RowMap map,
                     cudaStream_t stream) {
  if (n_rows <= 0) return DSA_OK;
  const bool vec = (row_bytes % 16 == 0) && (reinterpret_cast<uintptr_t>(src) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(dst) % 16 == 0);
  if (vec) {
    const int64_t cpr = row_bytes / 16;
    copy_rows_v16_kernel<RowMap><<<grid_for(n_rows * cpr, kUnroll), kThreads, 0, stream>>>(
        static_cast<const int4*>(src), static_cast<int4*>(dst), n_rows, cpr, map);
  } else {
    copy_rows_bytes_kernel<RowMap><<<grid_for(n_rows * row_bytes, 4), kThreads, 0, stream>>>(
        static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), n_rows, row_bytes, map);
  }
  DSA_CHECK_CUDA(cudaGetLastError());
  return DSA_OK;
}

}  // namespace

int64_t shard_len(int64_t n_tokens, int sp, int rank) {
  if (sp < 1 || rank < 0 || rank >= sp || n_tokens < 0) return -1;
  return n_tokens > rank ? (n_tokens - rank + sp - 1) / sp : 0;
}

int split_metadata(const int32_t* cu, int n_req, int64_t n_tokens, int sp, int rank,
                   int32_t* cu_shard, int32_t* pos, int32_t* bid, int32_t* gidx,
                   const void* src_rows, void* dst_rows, int64_t row_bytes,
                   cudaStream_t stream) {
  if (sp < 1 || rank < 0 || rank >= sp)
    return fail(DSA_ERR_INVALID, "split: need sp >= 1 and 0 <= rank < sp (sp=%d rank=%d)", sp,
                rank);
  if (n_req < 1 || n_tokens < 0 || n_tokens > INT32_MAX)
    return fail(DSA_ERR_INVALID, "split: need n_req >= 1 and 0 <= n_tokens < 2^31");
  if (!cu || !cu_shard) return fail(DSA_ERR_INVALID, "split: cu and cu_shard are required");
  const int64_t n_r = shard_len(n_tokens, sp, rank);
  if (n_r > 0 && (!pos || !bid))
    return fail(DSA_ERR_INVALID, "split: pos and bid are required when the shard is not empty");
  if (src_rows && (!dst_rows || row_bytes <= 0))
    return fail(DSA_ERR_INVALID, "split: a row gather needs dst_rows and row_bytes > 0");
  const int64_t meta_items = (n_r > n_req + 1) ? n_r : n_req + 1;
  split_meta_kernel<<<grid_for(meta_items, 1), kThreads, 0, stream>>>(cu, n_req, n_r, sp, rank,
                                                                      cu_shard, pos, bid, gidx);
  DSA_CHECK_CUDA(cudaGetLastError());
  if (src_rows) return launch_copy_rows(src_rows, dst_rows, n_r, row_bytes, SplitRows{sp, rank},
                                        stream);
  return DSA_OK;
}

int rerange(const void* gathered, void* out, int64_t n_tokens, int sp, int64_t rank_stride_rows,
            int64_t row_bytes, cudaStream_t stream) {
  if (sp < 1 || n_tokens < 0 || row_bytes <= 0 || rank_stride_rows < 0)
    return fail(DSA_ERR_INVALID, "rerange: need sp >= 1, n_tokens >= 0, row_bytes > 0");
  if (n_tokens == 0) return DSA_OK;
  if (!gathered || !out) return fail(DSA_ERR_INVALID, "rerange: null buffer");
  const int64_t need = (n_tokens + sp - 1) / sp;
  if (rank_stride_rows > 0 && rank_stride_rows < need)
    return fail(DSA_ERR_INVALID, "rerange: rank_stride_rows %lld < ceil(N/sp) = %lld",
                static_cast<long long>(rank_stride_rows), static_cast<long long>(need));
  RerangeRows map{sp, n_tokens / sp, n_tokens % sp, rank_stride_rows};
  return launch_copy_rows(gathered, out, n_tokens, row_bytes, map, stream);
}

cudaError_t split_read_errors(uint32_t* flags) { return read_and_clear_device_error(flags); }

}  // namespace dsa
