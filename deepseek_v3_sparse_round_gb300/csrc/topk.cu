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

#include "status.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kPerThread = 8;                       // consecutive entries per thread per chunk
constexpr int kChunk = kThreads * kPerThread;       // 4096 entries
constexpr int kBins = 2048;                         // 11-bit digits
constexpr int kStashKeys = 40960;                   // 160 KB of keys in shared memory
constexpr int kShortRow = 16384;                    // rows up to this length: kIn = 2

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;                     // -0.0 == +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

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

// kIn: 16-byte loads in flight per thread while the stash fills. Short rows (several CTAs per SM)
// take 2 and keep the registers for three CTAs per SM; long rows (one CTA per SM: the stash
// takes most of shared memory) take 4.
template <bool kStash, int kIn>
__global__ void __launch_bounds__(kThreads, kIn <= 2 ? 3 : 1)
topk_kernel(const float* __restrict__ scores, int64_t stride, const int32_t* __restrict__ pos,
            int k, int max_ctx, int32_t* __restrict__ topk) {
  extern __shared__ __align__(16) uint32_t stash[];
  __shared__ uint32_t hist[kBins];
  __shared__ uint32_t warp_tot[kWarps];
  __shared__ uint32_t s_digit, s_above;

  // Rows in reverse order: within a request of a round-robin shard, later rows are longer, so
  // the longest rows start first and the last CTAs to be scheduled get short ones.
  const int64_t t = static_cast<int64_t>(gridDim.x) - 1 - blockIdx.x;
  int32_t* out = topk + t * k;
  const int L = __ldg(pos + t) + 1;
  if (L < 1 || L > max_ctx) {
    if (threadIdx.x == 0) report_device_error(kErrBadLength);
    for (int j = threadIdx.x; j < k; j += kThreads) out[j] = -1;
    return;
  }
  if (L <= k) {                                     // every index is taken
    for (int j = threadIdx.x; j < k; j += kThreads) out[j] = j < L ? j : -1;
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
  uint32_t prefix = 0, prefix_mask = 0, remaining = static_cast<uint32_t>(k);
#pragma unroll 1
  for (int p = 0; p < 3; ++p) {
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
    // Thread j owns the 4 bins of mirror index m = kThreads-1-j, so an exclusive scan in thread
    // order counts every bin above them.
    const int m = kThreads - 1 - threadIdx.x;
    const uint32_t h0 = hist[4 * m], h1 = hist[4 * m + 1], h2 = hist[4 * m + 2],
                   h3 = hist[4 * m + 3];
    uint32_t tot;
    uint32_t above = block_exclusive_scan(h0 + h1 + h2 + h3, warp_tot, &tot);
    const uint32_t hs[4] = {h0, h1, h2, h3};
#pragma unroll
    for (int j = 3; j >= 0; --j) {
      if (above < remaining && above + hs[j] >= remaining) {
        s_digit = static_cast<uint32_t>(4 * m + j);
        s_above = above;
      }
      above += hs[j];
    }
    __syncthreads();
    remaining -= s_above;
    prefix |= s_digit << sh;
    prefix_mask |= dm << sh;
    __syncthreads();
  }
  const uint32_t T = prefix;
  const uint32_t need_eq = remaining;               // entries equal to T that are still taken
  const uint32_t n_gt = static_cast<uint32_t>(k) - remaining;

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
    for (int i = lo; i < hi; ++i) {
      const uint32_t key = stash[i];
      if (key > T) {
        out[g_before + (e_before < need_eq ? e_before : need_eq)] = i;
        ++g_before;
      } else if (key == T) {
        if (e_before < need_eq) out[g_before + e_before] = i;
        ++e_before;
      }
    }
    return;
  }
  uint32_t gt_done = 0, eq_done = 0;
  for (int base = 0; base < L && (gt_done < n_gt || eq_done < need_eq); base += kChunk) {
    uint32_t key[kPerThread];
    bool valid[kPerThread];
    load_keys<kStash>(row, stash, L, base, key, valid);
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
        out[g_before + (e_before < need_eq ? e_before : need_eq)] = i0 + j;
        ++g_before;
      } else if (key[j] == T) {
        if (e_before < need_eq) out[g_before + e_before] = i0 + j;
        ++e_before;
      }
    }
    gt_done += tot >> 16;
    eq_done += tot & 0xFFFFu;
  }
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
  if (max_ctx <= kStashKeys) {
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
