// Round-robin split metadata + row gather, and the rerange of an all-gathered buffer.
//
// "[DeepSeek v3.2] 上下文并行详解", section 2.B: rank r keeps the flattened tokens
// r, r+sp, r+2sp, ... and a metadata kernel recomputes cu_seqlens and batch indices after the
// scatter. Section 4 part 3 step B: the all-gathered rows arrive rank by rank and are put back
// in logical order. Both are plain HBM streams: 16-byte vector loads and stores over
// the flattened (row, 16-byte chunk) index space, several independent chunks in flight per
// thread, grid sized to a multiple of the SM count.
#include <cstdint>
#include <type_traits>
#include <cuda_runtime.h>

#include "status.cuh"

namespace dsa {

int num_sms_cached();
int64_t shard_len(int64_t n_tokens, int sp, int rank);

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
    if (static_cast<int64_t>(cu[mid]) <= g) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Source row of destination row `r` for the two copy patterns; the index arithmetic runs in
// the copy loop's index type (32-bit whenever the chunk count fits).
struct SplitRows {
  int sp, rank;
  template <typename I>
  __device__ __forceinline__ int64_t operator()(I t) const {
    return rank + static_cast<int64_t>(t) * sp;
  }
};
struct RerangeRows {
  int sp;
  int64_t per_rank;   // floor(N / sp) (packed) -- unused when padded
  int64_t rem;        // N % sp (packed)
  int64_t stride;     // > 0: padded blocks
  template <typename I>
  __device__ __forceinline__ int64_t operator()(I g) const {
    const I q = g % static_cast<I>(sp), j = g / static_cast<I>(sp);
    const int64_t qq = static_cast<int64_t>(q);
    const int64_t off = stride > 0 ? qq * stride : qq * per_rank + (qq < rem ? qq : rem);
    return off + static_cast<int64_t>(j);
  }
};

// Copy rows of 16-byte chunks: destination chunk i = (row i / cpr, chunk i % cpr) comes from
// source row map(row). Index math in Idx (32-bit whenever the chunk count fits), kUnroll
// independent 16-byte loads in flight per thread before their stores.
template <class RowMap, typename Idx>
__device__ __forceinline__ void copy_rows_body(const int4* __restrict__ src, int4* __restrict__ dst,
                                               Idx total, Idx cpr, RowMap map) {
  const Idx stride = static_cast<Idx>(gridDim.x) * blockDim.x;
  Idx i = static_cast<Idx>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + (kUnroll - 1) * stride < total; i += kUnroll * stride) {
    int4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const Idx cc = i + u * stride;
      const Idx r = cc / cpr;
      v[u] = ld_stream(src + map(r) * cpr + (cc - r * cpr));
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) st_stream(dst + (i + u * stride), v[u]);
  }
  for (; i < total; i += stride) {
    const Idx r = i / cpr;
    st_stream(dst + i, ld_stream(src + map(r) * cpr + (i - r * cpr)));
  }
}

template <class RowMap, typename Idx>
__global__ void __launch_bounds__(kThreads)
copy_rows_v16_kernel(const int4* __restrict__ src, int4* __restrict__ dst, int64_t n_rows,
                     int64_t chunks_per_row, RowMap map) {
  copy_rows_body<RowMap, Idx>(src, dst, static_cast<Idx>(n_rows * chunks_per_row),
                              static_cast<Idx>(chunks_per_row), map);
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

// Several tensors reranged by one launch: the flattened (tensor, row, 16-byte chunk) space of
// up to kMaxMulti tensors that share the row map, so one grid streams all of them (one ramp and
// one tail instead of one per tensor).
constexpr int kMaxMulti = 4;
// Unsigned division of n < 2^31 by a divisor fixed at launch: q = (n * m) >> shift with
// l = ceil(log2 d), shift = 31 + l, m = floor(2^shift / d) + 1 (< 2^32). The error term
// n * (m * d - 2^shift) / (d * 2^shift) stays below 1/d, so the floor is exact.
struct FastDiv {
  uint32_t d, m, shift;
  __device__ __forceinline__ uint32_t div(uint32_t n) const {
    return static_cast<uint32_t>((static_cast<uint64_t>(n) * m) >> shift);
  }
};
FastDiv make_fastdiv(uint32_t d) {
  uint32_t l = 0;
  while ((uint64_t(1) << l) < d) ++l;
  const uint32_t shift = 31 + l;
  return FastDiv{d, static_cast<uint32_t>((uint64_t(1) << shift) / d + 1), shift};
}

struct MultiRows {
  const int4* src[kMaxMulti];
  int4* dst[kMaxMulti];
  FastDiv cpr[kMaxMulti];          // 16-byte chunks per row
  uint32_t begin[kMaxMulti + 1];   // first flattened chunk of each tensor
  int n;
};

// Flattened (tensor, row, chunk) index space; each index's source row from the rerange map with
// the divisions by the chunk count and by sp done by multiply-shift (this loop issues about as
// many integer operations as it moves 16-byte chunks, so the divisions decide its rate).
__global__ void __launch_bounds__(kThreads)
rerange_multi_kernel(MultiRows mr, RerangeRows map, FastDiv fsp) {
  const uint32_t total = mr.begin[mr.n];
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t i0 = blockIdx.x * blockDim.x + threadIdx.x; i0 < total; i0 += kUnroll * stride) {
    int4 v[kUnroll];
    int4* d[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t i = i0 + u * stride;
      d[u] = nullptr;
      if (i < total) {
        int seg = 0;
#pragma unroll
        for (int q = 1; q < kMaxMulti; ++q) seg += (q < mr.n && i >= mr.begin[q]) ? 1 : 0;
        const uint32_t li = i - mr.begin[seg], cpr = mr.cpr[seg].d;
        const uint32_t r = mr.cpr[seg].div(li);
        const uint32_t j = fsp.div(r), rank = r - j * fsp.d;   // r = j * sp + rank
        const int64_t off = map.stride > 0
            ? static_cast<int64_t>(rank) * map.stride
            : static_cast<int64_t>(rank) * map.per_rank + (rank < map.rem ? rank : map.rem);
        v[u] = ld_stream(mr.src[seg] + (off + j) * cpr + (li - r * cpr));
        d[u] = mr.dst[seg] + li;
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (d[u] != nullptr) st_stream(d[u], v[u]);
  }
}

// One launch for the whole split: shard cu_seqlens (closed form), per-token metadata (the
// request found by binary search over cu staged in shared memory; positions offset by
// pos_base[b] when given, for a decode step's new tokens) and, when asked, the 16-byte row
// gather of the shard's tokens.
constexpr int kCuSmem = 4096;
template <bool kGather>
__global__ void __launch_bounds__(kThreads)
split_kernel(const int32_t* __restrict__ cu, const int32_t* __restrict__ pos_base, int n_req,
             int64_t n_r, int sp, int rank, int32_t* __restrict__ cu_shard,
             int32_t* __restrict__ pos, int32_t* __restrict__ bid, int32_t* __restrict__ gidx,
             const int4* __restrict__ src, int4* __restrict__ dst, int64_t chunks_per_row) {
  __shared__ int32_t s_cu[kCuSmem];
  const bool staged = n_req + 1 <= kCuSmem;
  if (staged) {
    for (int i = threadIdx.x; i <= n_req; i += blockDim.x) s_cu[i] = __ldg(cu + i);
    __syncthreads();
  }
  const int32_t* cuv = staged ? s_cu : cu;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (int64_t i = i0; i <= n_req; i += stride) cu_shard[i] = shard_count_below(cuv[i], sp, rank);
  for (int64_t t = i0; t < n_r; t += stride) {
    const int64_t g = rank + t * sp;
    const int b = find_request(cuv, n_req, g);
    pos[t] = static_cast<int32_t>(g - cuv[b] + (pos_base ? __ldg(pos_base + b) : 0));
    bid[t] = b;
    if (gidx) gidx[t] = static_cast<int32_t>(g);
  }
  if (kGather) {
    const int64_t total = n_r * chunks_per_row;
    if (total < (int64_t(1) << 31))
      copy_rows_body<SplitRows, uint32_t>(src, dst, static_cast<uint32_t>(total),
                                          static_cast<uint32_t>(chunks_per_row),
                                          SplitRows{sp, rank});
    else
      copy_rows_body<SplitRows, int64_t>(src, dst, total, chunks_per_row, SplitRows{sp, rank});
  }
}

// Paged KV-cache writes: row i of the source goes to the cache slot of its token. Two maps:
//   RerangeToCache  (the rerange fused with the cache write) i = logical token g, source row
//                   off[g % sp] + g / sp of the all-gathered buffer, slot s = g - cu[b];
//   LocalToCache    (a rank keeps only its own tokens) i = shard token t, g = rank + t * sp,
//                   source row t of the rank's local rows, slot j = t - cu_shard[b] (the
//                   token's index among request b's tokens on this rank).
// Slot x of request b is pool row block_table[b][x / page_size] * page_size + x % page_size.
// Chunks of the flattened (row, 16-byte chunk) space, kUnroll loads in flight per thread; the
// request of a token comes from a binary search over cu staged in shared memory. A token whose
// page is missing (negative entry, beyond max_pages or outside the pool) is skipped and
// recorded in the device error word.
struct PagedPool {
  const int32_t* table;
  int max_pages, page_size;
  int64_t pool_rows;
};

struct RerangeToCache {
  RerangeRows rows;
  template <typename I>
  __device__ __forceinline__ int64_t src(I i) const { return rows(i); }
  template <typename I>
  __device__ __forceinline__ int64_t token(I i) const { return static_cast<int64_t>(i); }
  template <typename I>
  __device__ __forceinline__ int64_t slot(I i, int32_t cu_b) const {
    return static_cast<int64_t>(i) - cu_b;
  }
};

struct LocalToCache {
  int sp, rank;
  template <typename I>
  __device__ __forceinline__ int64_t src(I i) const { return static_cast<int64_t>(i); }
  template <typename I>
  __device__ __forceinline__ int64_t token(I i) const {
    return rank + static_cast<int64_t>(i) * sp;
  }
  template <typename I>
  __device__ __forceinline__ int64_t slot(I i, int32_t cu_b) const {
    return static_cast<int64_t>(i) - shard_count_below(cu_b, sp, rank);
  }
};

template <typename Idx, int kBytes, class Map>
__global__ void __launch_bounds__(kThreads, 4)   // 4 CTAs per SM: enough loads in flight
paged_write_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ pool, Idx total,
                   Idx cpr, Map map, const int32_t* __restrict__ cu, int n_req, PagedPool pp) {
  using V = typename std::conditional<kBytes == 16, int4, uint8_t>::type;
  __shared__ int32_t s_cu[kCuSmem];
  const bool staged = n_req + 1 <= kCuSmem;
  if (staged) {
    for (int i = threadIdx.x; i <= n_req; i += blockDim.x) s_cu[i] = __ldg(cu + i);
    __syncthreads();
  }
  const int32_t* cuv = staged ? s_cu : cu;
  // largest power of two <= n_req - 1: the first step of the request search below
  int step0 = 0;
  if (n_req > 1) {
    step0 = 1;
    while (2 * step0 <= n_req - 1) step0 <<= 1;
  }
  const V* vs = reinterpret_cast<const V*>(src);
  V* vp = reinterpret_cast<V*>(pool);
  const Idx stride = static_cast<Idx>(gridDim.x) * blockDim.x;
  bool bad = false;
  for (Idx i = static_cast<Idx>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += kUnroll * stride) {
    // The source chunks do not depend on the page map: their loads go out first and are in
    // flight while the destinations are worked out.
    Idx r[kUnroll], c[kUnroll];
    int64_t g[kUnroll];
    bool in[kUnroll];
    V v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const Idx cc = i + u * stride;
      in[u] = cc < total;
      const Idx ci = in[u] ? cc : 0;
      r[u] = ci / cpr;
      c[u] = ci - r[u] * cpr;
      g[u] = map.token(r[u]);
      if constexpr (kBytes == 16) v[u] = ld_stream(vs + map.src(r[u]) * cpr + c[u]);
      else v[u] = vs[map.src(r[u]) * cpr + c[u]];
    }
    // Request of each chunk: the largest b < n_req with cu[b] <= g, by a fixed sequence of
    // halving steps (the same count for every thread), the kUnroll searches side by side.
    int b[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) b[u] = 0;
    for (int step = step0; step > 0; step >>= 1) {
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int t = b[u] + step;
        if (t < n_req && static_cast<int64_t>(cuv[t]) <= g[u]) b[u] = t;
      }
    }
    int64_t dst[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      // slot in the request's cache (cu is int32, so it fits 32 bits), its page and row
      const int x = static_cast<int>(map.slot(r[u], cuv[b[u]]));
      const int pi = x / pp.page_size;
      const int page = (in[u] && pi < pp.max_pages)
                           ? __ldg(pp.table + static_cast<int64_t>(b[u]) * pp.max_pages + pi)
                           : -1;
      const int64_t row = page < 0 ? -1 : static_cast<int64_t>(page) * pp.page_size + (x - pi * pp.page_size);
      dst[u] = (row >= 0 && row < pp.pool_rows) ? row * static_cast<int64_t>(cpr) + c[u] : -1;
      bad |= in[u] && dst[u] < 0;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (dst[u] < 0) continue;
      if constexpr (kBytes == 16) st_stream(vp + dst[u], v[u]);
      else vp[dst[u]] = v[u];
    }
  }
  if (bad) report_device_error(kErrBadIndex);
}

int num_sms() { return num_sms_cached(); }

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
    if (n_rows * cpr < (int64_t(1) << 31))
      copy_rows_v16_kernel<RowMap, uint32_t><<<grid_for(n_rows * cpr, kUnroll), kThreads, 0,
                                               stream>>>(
          static_cast<const int4*>(src), static_cast<int4*>(dst), n_rows, cpr, map);
    else
      copy_rows_v16_kernel<RowMap, int64_t><<<grid_for(n_rows * cpr, kUnroll), kThreads, 0,
                                              stream>>>(
          static_cast<const int4*>(src), static_cast<int4*>(dst), n_rows, cpr, map);
  } else {
    copy_rows_bytes_kernel<RowMap><<<grid_for(n_rows * row_bytes, 4), kThreads, 0, stream>>>(
        static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), n_rows, row_bytes, map);
  }
  DSA_CHECK_CUDA(cudaGetLastError());
  return DSA_OK;
}

// Rows 0..n_rows-1 of `src` into their cache slots (16-byte vectors when both buffers and
// row_bytes are multiples of 16, else byte copies).
template <class Map>
int launch_paged_write(const void* src_rows, void* pool, int64_t n_rows, int64_t row_bytes,
                       const Map& map, const int32_t* cu, int n_req, const PagedPool& pp,
                       cudaStream_t stream) {
  const bool vec = (row_bytes % 16 == 0) && (reinterpret_cast<uintptr_t>(src_rows) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(pool) % 16 == 0);
  const int64_t cpr = vec ? row_bytes / 16 : row_bytes;
  const int64_t total = n_rows * cpr;
  const int grid = grid_for(total, kUnroll);
  const auto* src = static_cast<const uint8_t*>(src_rows);
  auto* dst = static_cast<uint8_t*>(pool);
  if (vec && total < (int64_t(1) << 31))
    paged_write_kernel<uint32_t, 16, Map><<<grid, kThreads, 0, stream>>>(
        src, dst, static_cast<uint32_t>(total), static_cast<uint32_t>(cpr), map, cu, n_req, pp);
  else if (vec)
    paged_write_kernel<int64_t, 16, Map><<<grid, kThreads, 0, stream>>>(src, dst, total, cpr, map,
                                                                        cu, n_req, pp);
  else
    paged_write_kernel<int64_t, 1, Map><<<grid, kThreads, 0, stream>>>(src, dst, total, cpr, map,
                                                                       cu, n_req, pp);
  DSA_CHECK_CUDA(cudaGetLastError());
  return DSA_OK;
}

}  // namespace

int64_t shard_len(int64_t n_tokens, int sp, int rank) {
  if (sp < 1 || rank < 0 || rank >= sp || n_tokens < 0) return -1;
  return n_tokens > rank ? (n_tokens - rank + sp - 1) / sp : 0;
}

int split_metadata(const int32_t* cu, const int32_t* pos_base, int n_req, int64_t n_tokens,
                   int sp, int rank, int32_t* cu_shard, int32_t* pos, int32_t* bid,
                   int32_t* gidx, const void* src_rows, void* dst_rows, int64_t row_bytes,
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
  const bool vec = src_rows && (row_bytes % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(src_rows) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(dst_rows) % 16 == 0);
  if (vec) {                                       // metadata + row gather in one launch
    const int64_t cpr = row_bytes / 16;
    const int64_t items = n_r * cpr > meta_items ? n_r * cpr : meta_items;
    split_kernel<true><<<grid_for(items, kUnroll), kThreads, 0, stream>>>(
        cu, pos_base, n_req, n_r, sp, rank, cu_shard, pos, bid, gidx, static_cast<const int4*>(src_rows),
        static_cast<int4*>(dst_rows), cpr);
    DSA_CHECK_CUDA(cudaGetLastError());
    return DSA_OK;
  }
  split_kernel<false><<<grid_for(meta_items, 1), kThreads, 0, stream>>>(
      cu, pos_base, n_req, n_r, sp, rank, cu_shard, pos, bid, gidx, nullptr, nullptr, 0);
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

int rerange_multi(const void* const* gathered, void* const* out, const int64_t* row_bytes,
                  int n_tensors, int64_t n_tokens, int sp, int64_t rank_stride_rows,
                  cudaStream_t stream) {
  if (n_tensors < 1 || n_tensors > kMaxMulti)
    return fail(DSA_ERR_INVALID, "rerange_multi: 1 to %d tensors (got %d)", kMaxMulti, n_tensors);
  if (!gathered || !out || !row_bytes) return fail(DSA_ERR_INVALID, "rerange_multi: null array");
  if (sp < 1 || n_tokens < 0 || rank_stride_rows < 0)
    return fail(DSA_ERR_INVALID, "rerange_multi: need sp >= 1, n_tokens >= 0");
  const int64_t need = (n_tokens + sp - 1) / sp;
  if (rank_stride_rows > 0 && rank_stride_rows < need)
    return fail(DSA_ERR_INVALID, "rerange_multi: rank_stride_rows %lld < ceil(N/sp) = %lld",
                static_cast<long long>(rank_stride_rows), static_cast<long long>(need));
  MultiRows mr{};
  mr.n = n_tensors;
  int64_t total = 0;
  for (int q = 0; q < n_tensors; ++q) {
    if (!gathered[q] || !out[q] || row_bytes[q] <= 0)
      return fail(DSA_ERR_INVALID, "rerange_multi: tensor %d has a null buffer or no bytes", q);
    if (row_bytes[q] % 16 || reinterpret_cast<uintptr_t>(gathered[q]) % 16 ||
        reinterpret_cast<uintptr_t>(out[q]) % 16)
      return fail(DSA_ERR_INVALID, "rerange_multi: tensor %d is not in 16-byte rows", q);
    mr.src[q] = static_cast<const int4*>(gathered[q]);
    mr.dst[q] = static_cast<int4*>(out[q]);
    mr.cpr[q] = make_fastdiv(static_cast<uint32_t>(row_bytes[q] / 16));
    mr.begin[q] = static_cast<uint32_t>(total);
    total += n_tokens * (row_bytes[q] / 16);
    if (total >= (int64_t(1) << 31))
      return fail(DSA_ERR_UNSUPPORTED, "rerange_multi: more than 2^31 chunks in one launch");
  }
  mr.begin[n_tensors] = static_cast<uint32_t>(total);
  if (total == 0) return DSA_OK;
  RerangeRows map{sp, n_tokens / sp, n_tokens % sp, rank_stride_rows};
  rerange_multi_kernel<<<grid_for(total, kUnroll), kThreads, 0, stream>>>(
      mr, map, make_fastdiv(static_cast<uint32_t>(sp)));
  DSA_CHECK_CUDA(cudaGetLastError());
  return DSA_OK;
}

int rerange_paged(const void* gathered, void* pool, int64_t pool_rows, int64_t n_tokens, int sp,
                  int64_t rank_stride_rows, int64_t row_bytes, const int32_t* cu, int n_req,
                  const int32_t* block_table, int max_pages, int page_size,
                  cudaStream_t stream) {
  if (sp < 1 || n_tokens < 0 || row_bytes <= 0 || rank_stride_rows < 0 || n_req < 1 ||
      page_size < 1 || max_pages < 1 || pool_rows < 0)
    return fail(DSA_ERR_INVALID,
                "rerange_paged: need sp >= 1, n_tokens >= 0, row_bytes > 0, n_req >= 1, "
                "page_size >= 1, max_pages >= 1");
  if (n_tokens > INT32_MAX) return fail(DSA_ERR_INVALID, "rerange_paged: n_tokens >= 2^31");
  if (n_tokens == 0) return DSA_OK;
  if (!gathered || !pool || !cu || !block_table)
    return fail(DSA_ERR_INVALID, "rerange_paged: null pointer");
  const int64_t need = (n_tokens + sp - 1) / sp;
  if (rank_stride_rows > 0 && rank_stride_rows < need)
    return fail(DSA_ERR_INVALID, "rerange_paged: rank_stride_rows %lld < ceil(N/sp) = %lld",
                static_cast<long long>(rank_stride_rows), static_cast<long long>(need));
  RerangeToCache map{RerangeRows{sp, n_tokens / sp, n_tokens % sp, rank_stride_rows}};
  PagedPool pp{block_table, max_pages, page_size, pool_rows};
  return launch_paged_write(gathered, pool, n_tokens, row_bytes, map, cu, n_req, pp, stream);
}

int cache_local_paged(const void* local_rows, void* pool, int64_t pool_rows, int64_t n_tokens,
                      int sp, int rank, int64_t row_bytes, const int32_t* cu, int n_req,
                      const int32_t* block_table, int max_pages, int page_size,
                      cudaStream_t stream) {
  if (sp < 1 || rank < 0 || rank >= sp)
    return fail(DSA_ERR_INVALID, "cache_local_paged: need sp >= 1 and 0 <= rank < sp (sp=%d "
                                 "rank=%d)", sp, rank);
  if (n_tokens < 0 || row_bytes <= 0 || n_req < 1 || page_size < 1 || max_pages < 1 ||
      pool_rows < 0)
    return fail(DSA_ERR_INVALID,
                "cache_local_paged: need n_tokens >= 0, row_bytes > 0, n_req >= 1, "
                "page_size >= 1, max_pages >= 1");
  if (n_tokens > INT32_MAX) return fail(DSA_ERR_INVALID, "cache_local_paged: n_tokens >= 2^31");
  const int64_t n_r = shard_len(n_tokens, sp, rank);
  if (n_r == 0) return DSA_OK;
  if (!local_rows || !pool || !cu || !block_table)
    return fail(DSA_ERR_INVALID, "cache_local_paged: null pointer");
  PagedPool pp{block_table, max_pages, page_size, pool_rows};
  return launch_paged_write(local_rows, pool, n_r, row_bytes, LocalToCache{sp, rank}, cu, n_req,
                            pp, stream);
}

cudaError_t split_read_errors(uint32_t* flags) { return read_and_clear_device_error(flags); }

}  // namespace dsa
