// extern "C" entry points declared in include/dsa_rr.h: argument checks, error text, workspace
// sizing, and dispatch to the kernels of split.cu, topk.cu, indexer.cu and mla.cu.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <cuda_runtime.h>

#include "status.cuh"

namespace dsa {

// ---- defined in the kernel translation units ----
int64_t shard_len(int64_t n_tokens, int sp, int rank);
int split_metadata(const int32_t* cu, const int32_t* pos_base, int n_req, int64_t n_tokens,
                   int sp, int rank, int32_t* cu_shard, int32_t* pos, int32_t* bid, int32_t* gidx,
                   const void* src_rows, void* dst_rows, int64_t row_bytes, cudaStream_t stream);
int rerange(const void* gathered, void* out, int64_t n_tokens, int sp, int64_t rank_stride_rows,
            int64_t row_bytes, cudaStream_t stream);
size_t indexer_plan_bytes(int64_t n_q);
int indexer_scores(const void* q_idx, const float* w, const void* k_idx, int64_t n_kv_rows,
                   const int32_t* cu, const int32_t* pos, const int32_t* bid, int64_t n_q, int n_req,
                   int Hi, int Di, int max_ctx, const int32_t* block_table, int max_pages,
                   int page_size, float* scores, int64_t stride, void* ws, size_t ws_bytes,
                   uint32_t* hist, const float* q_scale, const float* k_scale, int skip_le,
                   cudaStream_t stream);
int quantize_fp8_rows(const void* x, int64_t rows, int cols, void* codes, float* scales,
                      cudaStream_t stream);
int quantize_fp8_latent(const void* c, int64_t rows, void* packed, cudaStream_t stream);
int dequantize_fp8_latent(const void* packed, int64_t rows, void* c, cudaStream_t stream);
int topk_select_hist(const float* scores, int64_t score_stride, const int32_t* pos, int64_t n_q,
                     int k, int max_ctx, const uint32_t* hist_rows, int32_t* topk,
                     cudaStream_t stream);
int topk_select(const float* scores, int64_t score_stride, const int32_t* pos, int64_t n_q, int k,
                int max_ctx, int32_t* topk, cudaStream_t stream);
int sparse_mla(const void* q, const void* c, int64_t n_kv_rows, const int32_t* cu, int n_req,
               const int32_t* bid, const int32_t* topk, int64_t n_q, int H, int dqk, int dv, int k,
               float scale, const int32_t* block_table, int max_pages, int page_size, void* o,
               float* lse, const int32_t* pos, void* ws, size_t ws_bytes, cudaStream_t stream);
size_t sparse_mla_workspace_bytes(int64_t n_q);
cudaError_t split_read_errors(uint32_t* flags);
int rerange_multi(const void* const* gathered, void* const* out, const int64_t* row_bytes,
                  int n_tensors, int64_t n_tokens, int sp, int64_t rank_stride_rows,
                  cudaStream_t stream);
int rerange_paged(const void* gathered, void* pool, int64_t pool_rows, int64_t n_tokens, int sp,
                  int64_t rank_stride_rows, int64_t row_bytes, const int32_t* cu, int n_req,
                  const int32_t* block_table, int max_pages, int page_size, cudaStream_t stream);
int cache_local_paged(const void* local_rows, void* pool, int64_t pool_rows, int64_t n_tokens,
                      int sp, int rank, int64_t row_bytes, const int32_t* cu, int n_req,
                      const int32_t* block_table, int max_pages, int page_size,
                      cudaStream_t stream);
int selftest_bounded_wait(long long limit_cycles, cudaStream_t stream);
cudaError_t selftest_read_errors(uint32_t* flags);
int probe_row_gather(const void* c, int64_t n_rows, const int32_t* rows, int n_ctas, int n_tiles,
                     int mode, int issuers, unsigned long long* cycles, cudaStream_t stream);
cudaError_t probe_read_errors(uint32_t* flags);
cudaError_t topk_read_errors(uint32_t* flags);
cudaError_t indexer_read_errors(uint32_t* flags);
cudaError_t mla_read_errors(uint32_t* flags);

namespace {
thread_local char g_msg[512] = "no error";
}

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
}

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  snprintf(g_msg, sizeof(g_msg), "CUDA error %d (%s) in %s", static_cast<int>(e),
           cudaGetErrorString(e), what);
  return DSA_ERR_CUDA;
}

// SM count of the current device, looked up once per device ordinal (grids and persistent
// pairs are sized from it). Concurrent first calls may both query; they store the same value.
int num_sms_cached() {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev >= 0 && dev < kMaxDevices) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return 148;
  if (dev >= 0 && dev < kMaxDevices) cache[dev].store(sms, std::memory_order_relaxed);
  return sms;
}

static size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// dsa_indexer_topk fuses the two steps (the indexer histograms the first radix digit of every
// score it writes; the top-k reads each row once) when a row can be longer than this: shorter
// rows are selected from a shared-memory copy of the row at least as fast, without the
// histogram's memset and atomics.
constexpr int kFuseMinCtx = 8192;
constexpr size_t kHistRowBytes = 2048 * sizeof(uint32_t);

static size_t hist_bytes(int64_t n_q, int max_ctx) {
  return max_ctx > kFuseMinCtx ? static_cast<size_t>(n_q) * kHistRowBytes : 0;
}

}  // namespace dsa

#define DSA_EXPORT __attribute__((visibility("default")))

extern "C" {

DSA_EXPORT const char* dsa_last_error_string(void) { return dsa::g_msg; }

DSA_EXPORT int dsa_version(void) { return 1; }

DSA_EXPORT int dsa_read_device_errors(uint32_t* flags) {
  if (!flags) return dsa::fail(DSA_ERR_INVALID, "flags is NULL");
  *flags = 0;
  DSA_CHECK_CUDA(cudaDeviceSynchronize());
  DSA_CHECK_CUDA(dsa::split_read_errors(flags));
  DSA_CHECK_CUDA(dsa::topk_read_errors(flags));
  DSA_CHECK_CUDA(dsa::indexer_read_errors(flags));
  DSA_CHECK_CUDA(dsa::mla_read_errors(flags));
  DSA_CHECK_CUDA(dsa::selftest_read_errors(flags));
  DSA_CHECK_CUDA(dsa::probe_read_errors(flags));
  return DSA_OK;
}

DSA_EXPORT int dsa_selftest_bounded_wait(int64_t limit_cycles, dsa_stream_t stream) {
  if (limit_cycles < 1 || limit_cycles > (1ll << 40))
    return dsa::fail(DSA_ERR_INVALID, "selftest: limit_cycles must be in [1, 2^40]");
  return dsa::selftest_bounded_wait(static_cast<long long>(limit_cycles),
                                    reinterpret_cast<cudaStream_t>(stream));
}

DSA_EXPORT int dsa_probe_row_gather(const void* c, int64_t n_rows, const int32_t* rows, int n_ctas,
                                    int n_tiles, int mode, int issuers, uint64_t* cycles,
                                    dsa_stream_t stream) {
  if (c == nullptr || rows == nullptr || cycles == nullptr)
    return dsa::fail(DSA_ERR_INVALID, "probe: null pointer");
  if (n_rows < 1 || n_rows > (1ll << 31) - 1 || n_ctas < 1 || n_ctas > 65535 || n_tiles < 1 ||
      static_cast<int64_t>(n_ctas) * n_tiles * 48 > (1ll << 31) - 1)
    return dsa::fail(DSA_ERR_INVALID, "probe: need 1 <= n_rows < 2^31, 1 <= n_ctas <= 65535, "
                                      "n_tiles >= 1 and n_ctas * n_tiles * 48 < 2^31");
  if (mode < 0 || mode > 7) return dsa::fail(DSA_ERR_INVALID, "probe: mode is 0 to 7");
  if (mode == 3 && (n_ctas % 2) != 0)
    return dsa::fail(DSA_ERR_INVALID, "probe: mode 3 runs CTA pairs: n_ctas must be even");
  if (mode == 1 && (issuers < 1 || issuers > 32))
    return dsa::fail(DSA_ERR_INVALID, "probe: 1 <= issuers <= 32 for mode 1");
  if ((reinterpret_cast<uintptr_t>(c) & 15u) != 0)
    return dsa::fail(DSA_ERR_INVALID, "probe: c must be 16-byte aligned");
  return dsa::probe_row_gather(c, n_rows, rows, n_ctas, n_tiles, mode, issuers,
                               reinterpret_cast<unsigned long long*>(cycles),
                               reinterpret_cast<cudaStream_t>(stream));
}

DSA_EXPORT int64_t dsa_rr_shard_len(int64_t n_tokens, int sp, int rank) {
  return dsa::shard_len(n_tokens, sp, rank);
}

DSA_EXPORT int dsa_rr_split_metadata(const int32_t* cu, int n_req, int64_t n_tokens, int sp, int rank,
                          int32_t* cu_shard, int32_t* pos, int32_t* bid, int32_t* gidx,
                          const void* src_rows, void* dst_rows, int64_t row_bytes,
                          dsa_stream_t stream) {
  return dsa::split_metadata(cu, nullptr, n_req, n_tokens, sp, rank, cu_shard, pos, bid, gidx,
                             src_rows, dst_rows, row_bytes, reinterpret_cast<cudaStream_t>(stream));
}

DSA_EXPORT int dsa_rr_split_decode_metadata(const int32_t* cu_new, const int32_t* pos_base,
                                            int n_req, int64_t n_tokens, int sp, int rank,
                                            int32_t* cu_shard, int32_t* pos, int32_t* bid,
                                            int32_t* gidx, const void* src_rows, void* dst_rows,
                                            int64_t row_bytes, dsa_stream_t stream) {
  if (!pos_base) return dsa::fail(DSA_ERR_INVALID, "split_decode: pos_base is required");
  return dsa::split_metadata(cu_new, pos_base, n_req, n_tokens, sp, rank, cu_shard, pos, bid,
                             gidx, src_rows, dst_rows, row_bytes,
                             reinterpret_cast<cudaStream_t>(stream));
}

DSA_EXPORT int dsa_rr_rerange(const void* gathered, void* out, int64_t n_tokens, int sp,
                   int64_t rank_stride_rows, int64_t row_bytes, dsa_stream_t stream) {
  return dsa::rerange(gathered, out, n_tokens, sp, rank_stride_rows, row_bytes,
                      reinterpret_cast<cudaStream_t>(stream));
}

DSA_EXPORT int dsa_rr_rerange_multi(const void* const* gathered, void* const* out,
                                    const int64_t* row_bytes, int n_tensors, int64_t n_tokens,
                                    int sp, int64_t rank_stride_rows, dsa_stream_t stream) {
  return dsa::rerange_multi(gathered, out, row_bytes, n_tensors, n_tokens, sp, rank_stride_rows,
                            reinterpret_cast<cudaStream_t>(stream));
}

DSA_EXPORT int dsa_rr_rerange_paged(const void* gathered, void* pool, int64_t pool_rows,
                                    int64_t n_tokens, int sp, int64_t rank_stride_rows,
                                    int64_t row_bytes, const int32_t* cu, int n_req,
                                    const int32_t* block_table, int max_pages, int page_size,
                                    dsa_stream_t stream) {
  return dsa::rerange_paged(gathered, pool, pool_rows, n_tokens, sp, rank_stride_rows, row_bytes,
                            cu, n_req, block_table, max_pages, page_size,
                            reinterpret_cast<cudaStream_t>(stream));
}

DSA_EXPORT int dsa_rr_cache_local_paged(const void* local_rows, void* pool, int64_t pool_rows,
                                        int64_t n_tokens, int sp, int rank, int64_t row_bytes,
                                        const int32_t* cu, int n_req, const int32_t* block_table,
                                        int max_pages, int page_size, dsa_stream_t stream) {
  return dsa::cache_local_paged(local_rows, pool, pool_rows, n_tokens, sp, rank, row_bytes, cu,
                                n_req, block_table, max_pages, page_size,
                                reinterpret_cast<cudaStream_t>(stream));
}

DSA_EXPORT int64_t dsa_score_row_stride(int max_ctx) {
  if (max_ctx < 1) return 0;
  return static_cast<int64_t>((max_ctx + 3) / 4) * 4;
}

DSA_EXPORT size_t dsa_indexer_topk_workspace_size(int64_t n_q, int max_ctx, int k) {
  (void)k;
  if (n_q < 0 || max_ctx < 1) return 0;
  const size_t plan = dsa::indexer_plan_bytes(n_q);
  const size_t scores = static_cast<size_t>(n_q) * static_cast<size_t>(dsa_score_row_stride(max_ctx)) *
                        sizeof(float);
  return dsa::round_up(plan, 256) + dsa::round_up(scores, 256) +
         dsa::round_up(dsa::hist_bytes(n_q, max_ctx), 256);
}

DSA_EXPORT int dsa_indexer_scores(const void* q_idx, const float* w, const void* k_idx, int64_t n_kv_rows,
                       const int32_t* cu, int n_req, const int32_t* pos, const int32_t* bid,
                       int64_t n_q, int Hi, int Di, int max_ctx, const int32_t* block_table,
                       int max_pages, int page_size, float* scores, int64_t score_stride,
                       void* workspace, size_t workspace_bytes, dsa_stream_t stream) {
  if (n_req < 1) return dsa::fail(DSA_ERR_INVALID, "indexer: n_req must be >= 1");
  if (score_stride % 4 != 0 || reinterpret_cast<uintptr_t>(scores) % 16 != 0)
    return dsa::fail(DSA_ERR_INVALID, "indexer: score rows must be 16-byte aligned");
  return dsa::indexer_scores(q_idx, w, k_idx, n_kv_rows, cu, pos, bid, n_q, n_req, Hi, Di,
                             max_ctx, block_table, max_pages, page_size, scores, score_stride,
                             workspace, workspace_bytes, nullptr, nullptr, nullptr, 0,
                             reinterpret_cast<cudaStream_t>(stream));
}

DSA_EXPORT int dsa_topk_select(const float* scores, int64_t score_stride, const int32_t* pos, int64_t n_q,
                    int k, int max_ctx, int32_t* topk, dsa_stream_t stream) {
  return dsa::topk_select(scores, score_stride, pos, n_q, k, max_ctx, topk,
                          reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace dsa {

// Indexer scores (bf16 rows, or FP8 rows with their scales) into the workspace's score rows,
// then the per-query top-k; fused through the first-digit histograms for long rows.
static int indexer_topk_impl(const void* q_idx, const float* q_scale, const float* w,
                             const void* k_idx, const float* k_scale, int64_t n_kv_rows,
                             const int32_t* cu, int n_req, const int32_t* pos, const int32_t* bid,
                             int64_t n_q, int Hi, int Di, int k, int max_ctx,
                             const int32_t* block_table, int max_pages, int page_size,
                             int32_t* topk, void* workspace, size_t workspace_bytes,
                             cudaStream_t stream) {
  if (n_q < 0 || max_ctx < 1 || k < 1)
    return fail(DSA_ERR_INVALID, "indexer_topk: need n_q >= 0, max_ctx >= 1, k >= 1");
  if (n_q == 0) return DSA_OK;
  const size_t need = dsa_indexer_topk_workspace_size(n_q, max_ctx, k);
  if (!workspace || workspace_bytes < need)
    return fail(DSA_ERR_WORKSPACE, "indexer_topk: workspace of %zu bytes < %zu",
                workspace_bytes, need);
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return fail(DSA_ERR_INVALID, "indexer_topk: workspace must be 256-byte aligned");
  if (n_req < 1) return fail(DSA_ERR_INVALID, "indexer: n_req must be >= 1");
  if (!topk) return fail(DSA_ERR_INVALID, "topk: null pointer");
  const size_t plan = round_up(indexer_plan_bytes(n_q), 256);
  float* scores = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + plan);
  const int64_t stride = dsa_score_row_stride(max_ctx);
  const size_t score_bytes =
      round_up(static_cast<size_t>(n_q) * static_cast<size_t>(stride) * sizeof(float), 256);
  uint32_t* hist = hist_bytes(n_q, max_ctx) > 0
                       ? reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) + plan +
                                                     score_bytes)
                       : nullptr;
  // A query whose history holds at most k keys selects all of them, so the top-k reads no score
  // of it: its group of queries is left out of the indexer when every query in it is such.
  int rc = indexer_scores(q_idx, w, k_idx, n_kv_rows, cu, pos, bid, n_q, n_req, Hi, Di, max_ctx,
                          block_table, max_pages, page_size, scores, stride, workspace, plan,
                          hist, q_scale, k_scale, k, stream);
  if (rc) return rc;
  if (hist == nullptr) return topk_select(scores, stride, pos, n_q, k, max_ctx, topk, stream);
  return topk_select_hist(scores, stride, pos, n_q, k, max_ctx, hist, topk, stream);
}

}  // namespace dsa

extern "C" {

DSA_EXPORT int dsa_indexer_topk(const void* q_idx, const float* w, const void* k_idx, int64_t n_kv_rows,
                     const int32_t* cu, int n_req, const int32_t* pos, const int32_t* bid,
                     int64_t n_q, int Hi, int Di, int k, int max_ctx, const int32_t* block_table,
                     int max_pages, int page_size, int32_t* topk, void* workspace,
                     size_t workspace_bytes, dsa_stream_t stream) {
  return dsa::indexer_topk_impl(q_idx, nullptr, w, k_idx, nullptr, n_kv_rows, cu, n_req, pos,
                                bid, n_q, Hi, Di, k, max_ctx, block_table, max_pages, page_size,
                                topk, workspace, workspace_bytes,
                                reinterpret_cast<cudaStream_t>(stream));
}

DSA_EXPORT int dsa_quantize_fp8_rows(const void* x, int64_t rows, int cols, void* codes,
                                     float* scales, dsa_stream_t stream) {
  return dsa::quantize_fp8_rows(x, rows, cols, codes, scales,
                                reinterpret_cast<cudaStream_t>(stream));
}

DSA_EXPORT int dsa_quantize_fp8_latent(const void* c, int64_t rows, void* packed,
                                       dsa_stream_t stream) {
  return dsa::quantize_fp8_latent(c, rows, packed, reinterpret_cast<cudaStream_t>(stream));
}

DSA_EXPORT int dsa_dequantize_fp8_latent(const void* packed, int64_t rows, void* c,
                                         dsa_stream_t stream) {
  return dsa::dequantize_fp8_latent(packed, rows, c, reinterpret_cast<cudaStream_t>(stream));
}

DSA_EXPORT int dsa_indexer_scores_fp8(const void* q8, const float* q_scale, const float* w,
                                      const void* k8, const float* k_scale, int64_t n_kv_rows,
                                      const int32_t* cu, int n_req, const int32_t* pos,
                                      const int32_t* bid, int64_t n_q, int Hi, int Di,
                                      int max_ctx, const int32_t* block_table, int max_pages,
                                      int page_size, float* scores, int64_t score_stride,
                                      void* workspace, size_t workspace_bytes,
                                      dsa_stream_t stream) {
  if (n_req < 1) return dsa::fail(DSA_ERR_INVALID, "indexer: n_req must be >= 1");
  if (!q_scale || !k_scale) return dsa::fail(DSA_ERR_INVALID, "indexer: FP8 scales are required");
  if (score_stride % 4 != 0 || reinterpret_cast<uintptr_t>(scores) % 16 != 0)
    return dsa::fail(DSA_ERR_INVALID, "indexer: score rows must be 16-byte aligned");
  return dsa::indexer_scores(q8, w, k8, n_kv_rows, cu, pos, bid, n_q, n_req, Hi, Di, max_ctx,
                             block_table, max_pages, page_size, scores, score_stride, workspace,
                             workspace_bytes, nullptr, q_scale, k_scale, 0,
                             reinterpret_cast<cudaStream_t>(stream));
}

DSA_EXPORT int dsa_indexer_topk_fp8(const void* q8, const float* q_scale, const float* w,
                                    const void* k8, const float* k_scale, int64_t n_kv_rows,
                                    const int32_t* cu, int n_req, const int32_t* pos,
                                    const int32_t* bid, int64_t n_q, int Hi, int Di, int k,
                                    int max_ctx, const int32_t* block_table, int max_pages,
                                    int page_size, int32_t* topk, void* workspace,
                                    size_t workspace_bytes, dsa_stream_t stream) {
  if (!q_scale || !k_scale) return dsa::fail(DSA_ERR_INVALID, "indexer: FP8 scales are required");
  return dsa::indexer_topk_impl(q8, q_scale, w, k8, k_scale, n_kv_rows, cu, n_req, pos, bid,
                                n_q, Hi, Di, k, max_ctx, block_table, max_pages, page_size, topk,
                                workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

DSA_EXPORT int dsa_sparse_mla(const void* q, const void* c, int64_t n_kv_rows, const int32_t* cu, int n_req,
                   const int32_t* bid, const int32_t* topk, int64_t n_q, int H, int dqk, int dv,
                   int k, float scale, const int32_t* block_table, int max_pages, int page_size,
                   void* o, float* lse, dsa_stream_t stream) {
  return dsa::sparse_mla(q, c, n_kv_rows, cu, n_req, bid, topk, n_q, H, dqk, dv, k, scale,
                         block_table, max_pages, page_size, o, lse, nullptr, nullptr, 0,
                         reinterpret_cast<cudaStream_t>(stream));
}

DSA_EXPORT size_t dsa_sparse_mla_workspace_size(int64_t n_q) {
  return dsa::sparse_mla_workspace_bytes(n_q);
}

DSA_EXPORT int dsa_sparse_mla_balanced(const void* q, const void* c, int64_t n_kv_rows,
                                       const int32_t* cu, int n_req, const int32_t* bid,
                                       const int32_t* pos, const int32_t* topk, int64_t n_q, int H,
                                       int dqk, int dv, int k, float scale,
                                       const int32_t* block_table, int max_pages, int page_size,
                                       void* o, float* lse, void* workspace,
                                       size_t workspace_bytes, dsa_stream_t stream) {
  if (pos == nullptr) return dsa::fail(DSA_ERR_INVALID, "mla: pos is required");
  return dsa::sparse_mla(q, c, n_kv_rows, cu, n_req, bid, topk, n_q, H, dqk, dv, k, scale,
                         block_table, max_pages, page_size, o, lse, pos, workspace,
                         workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
