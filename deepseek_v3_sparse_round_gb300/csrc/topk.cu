// Per-query top-k of fp32 score rows: radix select, lowest index wins ties, output ascending.
//
// "[RFC]: Parallel strategy for Deepseek v3.2 like models" (comments): the indexer selects the
// history top-K keys of each query. One CTA per query row. Scores become order-preserving
// 32-bit keys (-0.0 folded onto +0.0); three histogram passes (11, 11, 10 bits, most
// significant first) pin the exact k-th largest key T and how many entries equal to T still
// belong to the result; a final ordered pass writes every index with key > T and the lowest-
// index entries with key == T, in ascending index order, using block-wide prefix counts.
// Rows up to kStashKeys entries are read from global memory once and kept in shared memory;
// longer rows are re-read from global memory (L2) in every pass.
// Shared-memory access: the histogram passes read the stash with consecutive lanes on
// consecutive words (order does not matter for a histogram); the ordered pass gives each thread
// one contiguous, odd-length segment of the row, so a single block-wide scan orders the output
// and the lanes' reads still fall in distinct banks.
#include <cstdint>
#include <cuda_runtime.h>

#include "keys.cuh"
#include "status.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kPerThread = 8;                       // consecutive entries per thread per chunk
constexpr int kChunk = kThreads * kPerThread;       // 4096 entries
constexpr int kBins = kHistBins;                    // 11-bit digits
constexpr int kStashKeys = 40960;                   // 160 KB of keys in shared memory
constexpr int kShortRow = 16384;                    // rows up to this length: kIn = 2


// Exclusive prefix sum over threads in threadIdx order; returns the block total in *total.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* warp_tot,
                                                         uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < kWarps ? warp_tot[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kWarps) warp_tot[lane] = w;          // inclusive warp prefixes
  }
  __syncthreads();
  const uint32_t before = (warp > 0 ? warp_tot[warp - 1] : 0u) + x - v;
  *total = warp_tot[kWarps - 1];
  __syncthreads();                                  // warp_tot is reused by the next call
  return before;
}

template <bool kStash>
__device__ __forceinline__ void load_keys(const float* __restrict__ row, const uint32_t* stash,
                                          int L, int base, uint32_t (&key)[kPerThread],
                                          bool (&valid)[kPerThread]) {
  const int i0 = base + threadIdx.x * kPerThread;
  if (kStash) {
    if (i0 + kPerThread <= L) {                     // two 16-byte reads (i0 is a multiple of 8)
      const uint4 a = *reinterpret_cast<const uint4*>(stash + i0);
      const uint4 b = *reinterpret_cast<const uint4*>(stash + i0 + 4);
      key[0] = a.x; key[1] = a.y; key[2] = a.z; key[3] = a.w;
      key[4] = b.x; key[5] = b.y; key[6] = b.z; key[7] = b.w;
#pragma unroll
      for (int j = 0; j < kPerThread; ++j) valid[j] = true;
    } else {
#pragma unroll
      for (int j = 0; j < kPerThread; ++j) {
        valid[j] = i0 + j < L;
        key[j] = valid[j] ? stash[i0 + j] : 0u;
      }
    }
  } else {
    if (i0 + kPerThread <= L) {
      const float4 a = __ldcg(reinterpret_cast<const float4*>(row + i0));
      const float4 b = __ldcg(reinterpret_cast<const float4*>(row + i0 + 4));
      const float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (int j = 0; j < kPerThread; ++j) { key[j] = order_key(f[j]); valid[j] = true; }
    } else {
#pragma unroll
      for (int j = 0; j < kPerThread; ++j) {
        valid[j] = i0 + j < L;
        key[j] = valid[j] ? order_key(__ldcg(row + i0 + j)) : 0u;
      }
    }
  }
}

// The histogram passes do not depend on which thread sees which entry: from the stash they read
// entry base + j * kThreads + threadIdx.x, so the 32 lanes of a warp read 32 consecutive words
// (no bank conflicts); from global memory they use the blocked layout (16-byte loads).
template <bool kStash>
__device__ __forceinline__ void load_keys_any_order(const float* __restrict__ row,
                                                    const uint32_t* stash, int L, int base,
                                                    uint32_t (&key)[kPerThread],
                                                    bool (&valid)[kPerThread]) {
  if (kStash) {
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) {
      const int i = base + j * kThreads + static_cast<int>(threadIdx.x);
      valid[j] = i < L;
      key[j] = valid[j] ? stash[i] : 0u;
    }
  } else {
    load_keys<false>(row, stash, L, base, key, valid);
  }
}

// Digit of the bin holding the `remaining`-th largest entry of a filled histogram, and the
// number of entries in the bins above it (written to *s_digit / *s_above; all threads see them
// after the call). Thread j owns the 4 bins of mirror index m = kThreads-1-j, so an exclusive
// scan in thread order counts every bin above them.
__device__ __forceinline__ void pick_bin(const uint32_t* hist, uint32_t remaining,
                                         uint32_t* warp_tot, uint32_t* s_digit,
                                         uint32_t* s_above) {
  if (threadIdx.x == 0) {          // defined even if the counts fall short of `remaining`
    *s_digit = 0u;
    *s_above = 0u;
  }                                // (ordered before the writes below by the scan's barrier)
  const int m = kThreads - 1 - threadIdx.x;
  const uint32_t h0 = hist[4 * m], h1 = hist[4 * m + 1], h2 = hist[4 * m + 2],
                 h3 = hist[4 * m + 3];
  uint32_t tot;
  uint32_t above = block_exclusive_scan(h0 + h1 + h2 + h3, warp_tot, &tot);
  const uint32_t hs[4] = {h0, h1, h2, h3};
#pragma unroll
  for (int j = 3; j >= 0; --j) {
    if (above < remaining && above + hs[j] >= remaining) {
      *s_digit = static_cast<uint32_t>(4 * m + j);
      *s_above = above;
    }
    above += hs[j];
  }
  __syncthreads();
}

// Radix passes (11, 11, 10 bits, most significant first) from pass `first` on, over the keys
// whose top bits already match `prefix` under `prefix_mask`, finding the exact key T of the
// `remaining`-th largest of them and how many entries equal to T still belong to the result.
template <bool kStash>
__device__ __forceinline__ void radix_threshold(const float* __restrict__ row,
                                                const uint32_t* stash, int L, int k, int first,
                                                uint32_t prefix, uint32_t prefix_mask,
                                                uint32_t remaining, uint32_t* hist,
                                                uint32_t* warp_tot, uint32_t* s_digit,
                                                uint32_t* s_above, uint32_t* T_out,
                                                uint32_t* need_eq_out) {
  (void)k;
#pragma unroll 1
  for (int p = first; p < 3; ++p) {
    for (int b = threadIdx.x; b < kBins; b += kThreads) hist[b] = 0;
    __syncthreads();
    const int sh = p == 0 ? 21 : (p == 1 ? 10 : 0);
    const uint32_t dm = p == 2 ? 0x3FFu : 0x7FFu;
    for (int base = 0; base < L; base += kChunk) {
      uint32_t key[kPerThread];
      bool valid[kPerThread];
      load_keys_any_order<kStash>(row, stash, L, base, key, valid);
#pragma unroll
      for (int j = 0; j < kPerThread; ++j)
        if (valid[j] && (key[j] & prefix_mask) == prefix) atomicAdd(&hist[(key[j] >> sh) & dm], 1u);
    }
    __syncthreads();
    pick_bin(hist, remaining, warp_tot, s_digit, s_above);
    remaining -= *s_above;
    prefix |= *s_digit << sh;
    prefix_mask |= dm << sh;
    // the bin holds exactly the entries still to take: every key at or above its lowest key
    const bool done = p < 2 && hist[*s_digit] == remaining && prefix != 0u;
    __syncthreads();
    if (done) {
      *T_out = prefix - 1u;
      *need_eq_out = 0u;
      return;
    }
  }
  *T_out = prefix;
  *need_eq_out = remaining;
}

// Output of a row: k int32 indices. Writing them with 16-byte stores needs k % 4 == 0 and a
// 16-byte aligned row (the caller's topk pointer is only known to be 4-byte aligned).
__device__ __forceinline__ bool wide_out(const int32_t* out, int k) {
  return (k & 3) == 0 && (reinterpret_cast<uintptr_t>(out) & 15u) == 0;
}

// out[j] = j < n ? j : -1 for j < k (every index of a row of n <= k entries; n = 0: none).
__device__ __forceinline__ void fill_taken(int32_t* out, int k, int n, int n_threads) {
  if (wide_out(out, k)) {
    for (int j = static_cast<int>(threadIdx.x) * 4; j < k; j += n_threads * 4)
      *reinterpret_cast<int4*>(out + j) = make_int4(j < n ? j : -1, j + 1 < n ? j + 1 : -1,
                                                    j + 2 < n ? j + 2 : -1, j + 3 < n ? j + 3 : -1);
  } else {
    for (int j = static_cast<int>(threadIdx.x); j < k; j += n_threads) out[j] = j < n ? j : -1;
  }
}

// The ordered emission writes each selected index at its rank, a scattered 4-byte store. When
// the k indices fit the (then unused) 16-byte aligned histogram array and the row allows wide
// stores, they are ranked into that array instead and copied out with 16-byte stores.
__device__ __forceinline__ uint32_t* out_stage(uint32_t* hist, const int32_t* out, int k) {
  return k <= kBins && wide_out(out, k) ? hist : nullptr;
}
__device__ __forceinline__ void copy_stage(const uint32_t* stage, int32_t* out, int k,
                                           int n_threads) {
  __syncthreads();                                  // every rank written
  for (int j = static_cast<int>(threadIdx.x) * 4; j < k; j += n_threads * 4)
    *reinterpret_cast<int4*>(out + j) = *reinterpret_cast<const int4*>(stage + j);
}

// Ordered emission reading the row from global memory in chunks: every index with key > T and
// the lowest-index need_eq entries with key == T, in ascending index order (into `stage` when
// it is given, then copied to out).
__device__ __forceinline__ void emit_ordered_global(const float* __restrict__ row, int L,
                                                    uint32_t T, uint32_t need_eq, uint32_t n_gt,
                                                    int k, int32_t* __restrict__ out,
                                                    uint32_t* warp_tot, uint32_t* stage) {
  int32_t* dst = stage != nullptr ? reinterpret_cast<int32_t*>(stage) : out;
  uint32_t gt_done = 0, eq_done = 0;
  for (int base = 0; base < L && (gt_done < n_gt || eq_done < need_eq); base += kChunk) {
    uint32_t key[kPerThread];
    bool valid[kPerThread];
    load_keys<false>(row, nullptr, L, base, key, valid);
    uint32_t n_g = 0, n_e = 0;
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) {
      n_g += (valid[j] && key[j] > T);
      n_e += (valid[j] && key[j] == T);
    }
    uint32_t tot;
    const uint32_t before = block_exclusive_scan((n_g << 16) | n_e, warp_tot, &tot);
    uint32_t g_before = gt_done + (before >> 16), e_before = eq_done + (before & 0xFFFFu);
    const int i0 = base + threadIdx.x * kPerThread;
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) {
      if (!valid[j]) continue;
      if (key[j] > T) {
        dst[g_before + (e_before < need_eq ? e_before : need_eq)] = i0 + j;
        ++g_before;
      } else if (key[j] == T) {
        if (e_before < need_eq) dst[g_before + e_before] = i0 + j;
        ++e_before;
      }
    }
    gt_done += tot >> 16;
    eq_done += tot & 0xFFFFu;
  }
  if (stage != nullptr) copy_stage(stage, out, k, kThreads);
}

// kIn: 16-byte loads in flight per thread while the stash fills. Short rows (several CTAs per SM)
// take 2 and keep the registers for three CTAs per SM; long rows (one CTA per SM: the stash
// takes most of shared memory) take 4.
template <bool kStash, int kIn>
__global__ void __launch_bounds__(kThreads, kIn <= 2 ? 3 : 1)
topk_kernel(const float* __restrict__ scores, int64_t stride, const int32_t* __restrict__ pos,
            int k, int max_ctx, int32_t* __restrict__ topk) {
  extern __shared__ __align__(16) uint32_t stash[];
  __shared__ __align__(16) uint32_t hist[kBins];
  __shared__ uint32_t warp_tot[kWarps];
  __shared__ uint32_t s_digit, s_above;

  // Rows in reverse order: within a request of a round-robin shard, later rows are longer, so
  // the longest rows start first and the last CTAs to be scheduled get short ones.
  const int64_t t = static_cast<int64_t>(gridDim.x) - 1 - blockIdx.x;
  int32_t* out = topk + t * k;
  const int L = __ldg(pos + t) + 1;
  if (L < 1 || L > max_ctx) {
    if (threadIdx.x == 0) report_device_error(kErrBadLength);
    fill_taken(out, k, 0, kThreads);
    return;
  }
  if (L <= k) {                                     // every index is taken
    fill_taken(out, k, L, kThreads);
    return;
  }
  const float* row = scores + t * stride;

  if (kStash) {                                     // keys of the whole row into shared memory
    // four 16-byte loads in flight per thread, then their stores
    for (int i0 = threadIdx.x * 4; i0 < L; i0 += kThreads * 4 * kIn) {
      float4 v[kIn];
#pragma unroll
      for (int u = 0; u < kIn; ++u) {
        const int i = i0 + u * kThreads * 4;
        if (i + 4 <= L) v[u] = __ldcg(reinterpret_cast<const float4*>(row + i));
      }
#pragma unroll
      for (int u = 0; u < kIn; ++u) {
        const int i = i0 + u * kThreads * 4;
        if (i + 4 <= L) {
          *reinterpret_cast<uint4*>(stash + i) =
              make_uint4(order_key(v[u].x), order_key(v[u].y), order_key(v[u].z), order_key(v[u].w));
        } else {
          for (int j = i; j < L; ++j) stash[j] = order_key(__ldcg(row + j));
        }
      }
    }
  }

  // ---- three radix passes: find the exact k-th largest key T ----
  uint32_t T, need_eq;
  radix_threshold<kStash>(row, stash, L, k, 0, 0u, 0u, static_cast<uint32_t>(k), hist, warp_tot,
                          &s_digit, &s_above, &T, &need_eq);
  const uint32_t n_gt = static_cast<uint32_t>(k) - need_eq;

  // ---- ordered emission ----
  if (kStash) {
    // One contiguous segment of the row per thread (odd length, so the lanes' reads fall in
    // distinct banks), one block-wide scan of the per-thread counts, then every thread writes
    // its selected indices in order.
    const int seg = ((L + kThreads - 1) / kThreads) | 1;
    const int lo = min(static_cast<int>(threadIdx.x) * seg, L), hi = min(lo + seg, L);
    uint32_t n_g = 0, n_e = 0;
    for (int i = lo; i < hi; ++i) {
      const uint32_t key = stash[i];
      n_g += key > T;
      n_e += key == T;
    }
    uint32_t tot;                                   // counts < 2^16: L <= kStashKeys
    const uint32_t before = block_exclusive_scan((n_g << 16) | n_e, warp_tot, &tot);
    uint32_t g_before = before >> 16, e_before = before & 0xFFFFu;
    uint32_t* stage = out_stage(hist, out, k);
    int32_t* dst = stage != nullptr ? reinterpret_cast<int32_t*>(stage) : out;
    for (int i = lo; i < hi; ++i) {
      const uint32_t key = stash[i];
      if (key > T) {
        dst[g_before + (e_before < need_eq ? e_before : need_eq)] = i;
        ++g_before;
      } else if (key == T) {
        if (e_before < need_eq) dst[g_before + e_before] = i;
        ++e_before;
      }
    }
    if (stage != nullptr) copy_stage(stage, out, k, kThreads);
    return;
  }
  emit_ordered_global(row, L, T, need_eq, n_gt, k, out, warp_tot, out_stage(hist, out, k));
}

// ------------------------------------------------------------------------------------------
// Rows of at most kShortMax entries (batches whose longest row is that short): the same
// selection as topk_kernel<true, ...> with a 256-thread CTA per row, so that more rows are in
// flight per SM and every block-wide barrier spans 8 warps instead of 16; each thread owns 8
// histogram bins.
constexpr int kShortMax = 4096;
constexpr int kShortThreads = 256;
constexpr int kShortWarps = kShortThreads / 32;
constexpr int kShortBinsPerThread = kBins / kShortThreads;

__device__ __forceinline__ uint32_t short_block_scan(uint32_t v, uint32_t* warp_tot,
                                                     uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < kShortWarps ? warp_tot[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kShortWarps) warp_tot[lane] = w;
  }
  __syncthreads();
  const uint32_t before = (warp > 0 ? warp_tot[warp - 1] : 0u) + x - v;
  *total = warp_tot[kShortWarps - 1];
  __syncthreads();
  return before;
}

__global__ void __launch_bounds__(kShortThreads, 6)
topk_short_kernel(const float* __restrict__ scores, int64_t stride,
                  const int32_t* __restrict__ pos, int k, int max_ctx,
                  int32_t* __restrict__ topk) {
  __shared__ __align__(16) uint32_t stash[kShortMax];
  __shared__ __align__(16) uint32_t hist[kBins];
  __shared__ uint32_t warp_tot[kShortWarps];
  __shared__ uint32_t s_digit, s_above;
  const int64_t t = static_cast<int64_t>(gridDim.x) - 1 - blockIdx.x;   // longest rows first
  int32_t* out = topk + t * k;
  const int L = __ldg(pos + t) + 1;
  if (L < 1 || L > max_ctx || L > kShortMax) {
    if (threadIdx.x == 0) report_device_error(kErrBadLength);
    fill_taken(out, k, 0, kShortThreads);
    return;
  }
  if (L <= k) {
    fill_taken(out, k, L, kShortThreads);
    return;
  }
  const float* row = scores + t * stride;
  // the row's keys into shared memory: every thread's 16-byte loads issued before their stores
  {
    constexpr int kLoads = kShortMax / (kShortThreads * 4);   // 4
    float4 v[kLoads];
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
      const int i = (u * kShortThreads + static_cast<int>(threadIdx.x)) * 4;
      if (i + 4 <= L) v[u] = __ldcg(reinterpret_cast<const float4*>(row + i));
    }
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
      const int i = (u * kShortThreads + static_cast<int>(threadIdx.x)) * 4;
      if (i + 4 <= L) {
        *reinterpret_cast<uint4*>(stash + i) =
            make_uint4(order_key(v[u].x), order_key(v[u].y), order_key(v[u].z), order_key(v[u].w));
      } else {
        for (int j = i; j < L && j < i + 4; ++j) stash[j] = order_key(__ldcg(row + j));
      }
    }
  }
  // up to three radix passes over the stash (11, 11, 10 bits)
  uint32_t prefix = 0, prefix_mask = 0, remaining = static_cast<uint32_t>(k);
  bool whole_bin = false;                            // every entry of the final bin is taken
#pragma unroll 1
  for (int p = 0; p < 3; ++p) {
    for (int b = threadIdx.x; b < kBins; b += kShortThreads) hist[b] = 0;
    if (threadIdx.x == 0) { s_digit = 0u; s_above = 0u; }
    __syncthreads();
    const int sh = p == 0 ? 21 : (p == 1 ? 10 : 0);
    const uint32_t dm = p == 2 ? 0x3FFu : 0x7FFu;
    for (int i = threadIdx.x; i < L; i += kShortThreads) {
      const uint32_t key = stash[i];
      if ((key & prefix_mask) == prefix) atomicAdd(&hist[(key >> sh) & dm], 1u);
    }
    __syncthreads();
    // thread j owns the bins of mirror index m = kShortThreads-1-j, so the exclusive scan in
    // thread order counts every bin above them
    const int m = kShortThreads - 1 - static_cast<int>(threadIdx.x);
    uint32_t hs[kShortBinsPerThread], sum = 0;
#pragma unroll
    for (int q = 0; q < kShortBinsPerThread; ++q) {
      hs[q] = hist[kShortBinsPerThread * m + q];
      sum += hs[q];
    }
    uint32_t tot;
    uint32_t above = short_block_scan(sum, warp_tot, &tot);
#pragma unroll
    for (int q = kShortBinsPerThread - 1; q >= 0; --q) {
      if (above < remaining && above + hs[q] >= remaining) {
        s_digit = static_cast<uint32_t>(kShortBinsPerThread * m + q);
        s_above = above;
      }
      above += hs[q];
    }
    __syncthreads();
    remaining -= s_above;
    prefix |= s_digit << sh;
    prefix_mask |= dm << sh;
    // the bin holds exactly the entries still to take: all of them, no further pass
    const bool done = p < 2 && hist[s_digit] == remaining && prefix != 0u;
    __syncthreads();
    if (done) { whole_bin = true; break; }
  }
  // whole_bin: taken = every key at or above the bin's lowest key (its lower bits all zero)
  const uint32_t T = whole_bin ? prefix - 1u : prefix, need_eq = whole_bin ? 0u : remaining;
  // ordered emission: one contiguous odd-length segment per thread, one block-wide scan
  const int seg = ((L + kShortThreads - 1) / kShortThreads) | 1;
  const int lo = min(static_cast<int>(threadIdx.x) * seg, L), hi = min(lo + seg, L);
  uint32_t n_g = 0, n_e = 0;
  for (int i = lo; i < hi; ++i) {
    const uint32_t key = stash[i];
    n_g += key > T;
    n_e += key == T;
  }
  uint32_t tot;
  const uint32_t before = short_block_scan((n_g << 16) | n_e, warp_tot, &tot);
  uint32_t g_before = before >> 16, e_before = before & 0xFFFFu;
  uint32_t* stage = out_stage(hist, out, k);
  int32_t* dst = stage != nullptr ? reinterpret_cast<int32_t*>(stage) : out;
  for (int i = lo; i < hi; ++i) {
    const uint32_t key = stash[i];
    if (key > T) {
      dst[g_before + (e_before < need_eq ? e_before : need_eq)] = i;
      ++g_before;
    } else if (key == T) {
      if (e_before < need_eq) dst[g_before + e_before] = i;
      ++e_before;
    }
  }
  if (stage != nullptr) copy_stage(stage, out, k, kShortThreads);
}

// ------------------------------------------------------------------------------------------
// Top-k fed by the indexer's sampled first-digit histograms (the fused indexer -> top-k path).
//
// Rows of up to kCap entries are kept whole in shared memory (key and index). For longer rows
// the indexer epilogue counted, per query, the first radix digit (top 11 bits of the order key)
// of one score in kHistSample. From those counts the kernel takes the highest bin T0 above
// which the sample holds comfortably more than k / kHistSample scores (a margin of four
// standard deviations), so the entries with digit >= T0 very likely number at least k and only
// a few thousand. One pass over the row (prefetched into L2 at the start) keeps exactly those
// entries, compacted in index order; their exact count decides: between k and kCap, the three
// radix passes and the ordered emission run over that short list; otherwise (a sample that
// misled, or a crowded boundary) the row takes the global-memory passes. The result is exact
// either way; the sample only decides how much work it takes.
constexpr int kCap = 8192;                          // kept entries in shared memory (64 KB)
constexpr int kCompactPerLane = 16;                 // entries per lane per compaction chunk
constexpr int kCompactChunk = kThreads * kCompactPerLane;

__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__global__ void __launch_bounds__(kThreads, 2)
topk_hist_kernel(const float* __restrict__ scores, int64_t stride, const int32_t* __restrict__ pos,
                 int k, int max_ctx, const uint32_t* __restrict__ hist_rows,
                 int32_t* __restrict__ topk) {
  extern __shared__ __align__(16) uint32_t kept[];   // keys [kCap], then indices [kCap]
  __shared__ __align__(16) uint32_t hist[kBins];
  __shared__ uint32_t warp_tot[kWarps];
  __shared__ uint32_t s_digit, s_above;
  uint32_t* ckey = kept;
  uint32_t* cidx = kept + kCap;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  const int64_t t = static_cast<int64_t>(gridDim.x) - 1 - blockIdx.x;   // longest rows first
  int32_t* out = topk + t * k;
  const int L = __ldg(pos + t) + 1;
  if (L < 1 || L > max_ctx) {
    if (threadIdx.x == 0) report_device_error(kErrBadLength);
    fill_taken(out, k, 0, kThreads);
    return;
  }
  if (L <= k) {
    fill_taken(out, k, L, kThreads);
    return;
  }
  const float* row = scores + t * stride;
  if (threadIdx.x == 0) {                             // the row streams into L2 meanwhile
    const uint32_t bytes = static_cast<uint32_t>((L + 3) / 4) * 16u;
    for (uint32_t off = 0; off < bytes; off += 32768u)
      prefetch_l2_bulk(reinterpret_cast<const char*>(row) + off, min(32768u, bytes - off));
  }
  uint32_t T0 = 0;                                    // keep every entry (rows of <= kCap)
  if (L > kCap) {
    const uint4* h = reinterpret_cast<const uint4*>(hist_rows + t * kBins);
    for (int i = threadIdx.x; i < kBins / 4; i += kThreads)
      reinterpret_cast<uint4*>(hist)[i] = __ldcg(h + i);
    __syncthreads();
    const float mean = static_cast<float>(k) / kHistSample;
    const uint32_t need = static_cast<uint32_t>(ceilf(mean + 4.f * sqrtf(mean))) + 16u;
    pick_bin(hist, need, warp_tot, &s_digit, &s_above);   // bin 0 if the sample falls short
    T0 = s_digit;
    __syncthreads();
  }

  // ---- compaction: entries with digit >= T0, in index order. Warp w reads its
  // kCompactPerLane * 32 entries of a chunk in coalesced rounds of 32 lanes x 4; the per-warp
  // counts are scanned across the block, then each round is placed by a warp scan. Entries
  // beyond kCap are counted, not stored.
  uint32_t kept_so_far = 0;
  // this lane's 16 entries of chunk `base` (coalesced rounds of 32 lanes x 4), loaded one
  // chunk ahead of their use
  auto load_chunk = [&](int base, float4 (&v)[kCompactPerLane / 4]) {
    const int wb = base + warp * (kCompactPerLane * 32);
#pragma unroll
    for (int j = 0; j < kCompactPerLane / 4; ++j) {
      const int i = wb + 128 * j + 4 * lane;
      if (i + 4 <= L) {
        v[j] = __ldcg(reinterpret_cast<const float4*>(row + i));
      } else {
        v[j].x = i < L ? __ldcg(row + i) : 0.f;
        v[j].y = i + 1 < L ? __ldcg(row + i + 1) : 0.f;
        v[j].z = i + 2 < L ? __ldcg(row + i + 2) : 0.f;
        v[j].w = i + 3 < L ? __ldcg(row + i + 3) : 0.f;
      }
    }
  };
  float4 vnext[kCompactPerLane / 4];
  load_chunk(0, vnext);
  for (int base = 0; base < L; base += kCompactChunk) {
    const int wb = base + warp * (kCompactPerLane * 32);
    float4 vcur[kCompactPerLane / 4];
#pragma unroll
    for (int j = 0; j < kCompactPerLane / 4; ++j) vcur[j] = vnext[j];
    if (base + kCompactChunk < L) load_chunk(base + kCompactChunk, vnext);
    uint32_t key[kCompactPerLane / 4][4];
    uint32_t keepm[kCompactPerLane / 4];
    uint32_t cnt = 0;
#pragma unroll
    for (int j = 0; j < kCompactPerLane / 4; ++j) {
      const int i = wb + 128 * j + 4 * lane;
      const float f[4] = {vcur[j].x, vcur[j].y, vcur[j].z, vcur[j].w};
      uint32_t m = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        key[j][e] = order_key(f[e]);
        if (i + e < L && first_digit(key[j][e]) >= T0) m |= 1u << e;
      }
      keepm[j] = m;
      cnt += __popc(m);
    }
    const uint32_t warp_cnt = __reduce_add_sync(0xffffffffu, cnt);
    uint32_t tot;
    const uint32_t wbefore = block_exclusive_scan(lane == 0 ? warp_cnt : 0u, warp_tot, &tot);
    uint32_t at = kept_so_far + __shfl_sync(0xffffffffu, wbefore, 0);
#pragma unroll
    for (int j = 0; j < kCompactPerLane / 4; ++j) {
      const uint32_t c = __popc(keepm[j]);
      uint32_t incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      uint32_t dst = at + incl - c;
      const int i = wb + 128 * j + 4 * lane;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if ((keepm[j] & (1u << e)) && dst < static_cast<uint32_t>(kCap)) {
          ckey[dst] = key[j][e];
          cidx[dst] = static_cast<uint32_t>(i + e);
        }
        dst += (keepm[j] >> e) & 1u;
      }
      at += __shfl_sync(0xffffffffu, incl, 31);
    }
    kept_so_far += tot;
  }
  __syncthreads();
  uint32_t T, need_eq;
  if (kept_so_far > static_cast<uint32_t>(kCap) || kept_so_far < static_cast<uint32_t>(k)) {
    radix_threshold<false>(row, nullptr, L, k, 0, 0u, 0u, static_cast<uint32_t>(k), hist,
                           warp_tot, &s_digit, &s_above, &T, &need_eq);
    emit_ordered_global(row, L, T, need_eq, static_cast<uint32_t>(k) - need_eq, k, out, warp_tot,
                        out_stage(hist, out, k));
    return;
  }
  const int n = static_cast<int>(kept_so_far);

  // ---- three radix passes over the kept entries ----
  uint32_t prefix = 0, prefix_mask = 0;
  uint32_t remaining = static_cast<uint32_t>(k);
#pragma unroll 1
  for (int p = 0; p < 3; ++p) {
    for (int b = threadIdx.x; b < kBins; b += kThreads) hist[b] = 0;
    __syncthreads();
    const int sh = p == 0 ? 21 : (p == 1 ? 10 : 0);
    const uint32_t dm = p == 2 ? 0x3FFu : 0x7FFu;
    for (int i = threadIdx.x; i < n; i += kThreads) {
      const uint32_t key = ckey[i];
      if ((key & prefix_mask) == prefix) atomicAdd(&hist[(key >> sh) & dm], 1u);
    }
    __syncthreads();
    pick_bin(hist, remaining, warp_tot, &s_digit, &s_above);
    remaining -= s_above;
    prefix |= s_digit << sh;
    prefix_mask |= dm << sh;
    // the bin holds exactly the entries still to take: every key at or above its lowest key
    const bool done = p < 2 && hist[s_digit] == remaining && prefix != 0u;
    __syncthreads();
    if (done) {
      prefix -= 1u;
      remaining = 0u;
      break;
    }
  }
  T = prefix;
  need_eq = remaining;

  // ---- ordered emission over the kept list (already in index order) ----
  const int seg = ((n + kThreads - 1) / kThreads) | 1;
  const int lo = min(static_cast<int>(threadIdx.x) * seg, n), hi = min(lo + seg, n);
  uint32_t n_g = 0, n_e = 0;
  for (int i = lo; i < hi; ++i) {
    const uint32_t key = ckey[i];
    n_g += key > T;
    n_e += key == T;
  }
  uint32_t tot;                                       // counts < 2^16: n <= kCap
  const uint32_t before = block_exclusive_scan((n_g << 16) | n_e, warp_tot, &tot);
  uint32_t g_before = before >> 16, e_before = before & 0xFFFFu;
  uint32_t* stage = out_stage(hist, out, k);
  int32_t* dst = stage != nullptr ? reinterpret_cast<int32_t*>(stage) : out;
  for (int i = lo; i < hi; ++i) {
    const uint32_t key = ckey[i];
    if (key > T) {
      dst[g_before + (e_before < need_eq ? e_before : need_eq)] = static_cast<int32_t>(cidx[i]);
      ++g_before;
    } else if (key == T) {
      if (e_before < need_eq) dst[g_before + e_before] = static_cast<int32_t>(cidx[i]);
      ++e_before;
    }
  }
  if (stage != nullptr) copy_stage(stage, out, k, kThreads);
}

}  // namespace

int topk_select(const float* scores, int64_t score_stride, const int32_t* pos, int64_t n_q, int k,
                int max_ctx, int32_t* topk, cudaStream_t stream) {
  if (n_q < 0 || k < 1 || max_ctx < 1)
    return fail(DSA_ERR_INVALID, "topk: need n_q >= 0, k >= 1, max_ctx >= 1");
  if (n_q == 0) return DSA_OK;
  if (!scores || !pos || !topk) return fail(DSA_ERR_INVALID, "topk: null pointer");
  if (score_stride < max_ctx || score_stride % 4 != 0 ||
      reinterpret_cast<uintptr_t>(scores) % 16 != 0)
    return fail(DSA_ERR_INVALID, "topk: score_stride must be >= max_ctx, a multiple of 4, and "
                                 "scores 16-byte aligned");
  if (n_q > INT32_MAX) return fail(DSA_ERR_UNSUPPORTED, "topk: n_q too large");
  if (max_ctx <= kShortMax) {
    topk_short_kernel<<<static_cast<unsigned>(n_q), kShortThreads, 0, stream>>>(
        scores, score_stride, pos, k, max_ctx, topk);
  } else if (max_ctx <= kStashKeys) {
    const size_t smem = static_cast<size_t>(((max_ctx + 3) / 4) * 4) * sizeof(uint32_t);
    const int max_smem = kStashKeys * static_cast<int>(sizeof(uint32_t));
    if (max_ctx <= kShortRow) {
      DSA_CHECK_CUDA(cudaFuncSetAttribute(topk_kernel<true, 2>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem));
      topk_kernel<true, 2><<<static_cast<unsigned>(n_q), kThreads, smem, stream>>>(
          scores, score_stride, pos, k, max_ctx, topk);
    } else {
      DSA_CHECK_CUDA(cudaFuncSetAttribute(topk_kernel<true, 4>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem));
      topk_kernel<true, 4><<<static_cast<unsigned>(n_q), kThreads, smem, stream>>>(
          scores, score_stride, pos, k, max_ctx, topk);
    }
  } else {
    topk_kernel<false, 2><<<static_cast<unsigned>(n_q), kThreads, 0, stream>>>(
        scores, score_stride, pos, k, max_ctx, topk);
  }
  DSA_CHECK_CUDA(cudaGetLastError());
  return DSA_OK;
}

cudaError_t topk_read_errors(uint32_t* flags) { return read_and_clear_device_error(flags); }

}  // namespace dsa

namespace dsa {

// Top-k of rows whose sampled first-digit histograms (hist_rows [n_q, kHistBins] u32, counts of
// the scores at positions s <= pos_t with s % kHistSample == 0) the indexer produced.
int topk_select_hist(const float* scores, int64_t score_stride, const int32_t* pos, int64_t n_q,
                     int k, int max_ctx, const uint32_t* hist_rows, int32_t* topk,
                     cudaStream_t stream) {
  if (n_q == 0) return DSA_OK;
  if (n_q > INT32_MAX) return fail(DSA_ERR_UNSUPPORTED, "topk: n_q too large");
  const int smem = 2 * kCap * static_cast<int>(sizeof(uint32_t));
  DSA_CHECK_CUDA(cudaFuncSetAttribute(topk_hist_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  topk_hist_kernel<<<static_cast<unsigned>(n_q), kThreads, smem, stream>>>(
      scores, score_stride, pos, k, max_ctx, hist_rows, topk);
  DSA_CHECK_CUDA(cudaGetLastError());
  return DSA_OK;
}

}  // namespace dsa
