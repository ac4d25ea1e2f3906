// dsa_indexer_topk_noalloc: the indexer + top-k call for callers that cannot allocate device
// memory themselves.
//
// Who needs it: dsa_indexer_topk asks the caller for a scratch buffer (score rows plus a small
// schedule). Some callers cannot obtain one: a host framework that reserved all device memory
// in its own pool at start-up and allows no further cudaMalloc, a language runtime without a
// CUDA allocator binding, or a latency-critical serving loop that must not call cudaMalloc or
// cudaFree because those calls can synchronise the device. This entry point needs no buffer:
// its scratch is one file-scope __device__ array of DSA_NOALLOC_SCRATCH_BYTES (64 MiB), which
// every GPU that loads the library holds until the process exits.
//
// Set-up: the first call on a device (with that device current) looks up the array's device
// address with cudaGetSymbolAddress and caches it per device; make that first call before any
// stream capture. The host-side name of the array is only a stand-in, never passed to a kernel.
// Sharing: every call uses the same array and leaves the last call's contents in it. Nothing in
// it has to start at zero (the planning kernel rewrites the schedule and the indexer writes
// every score the top-k reads), but calls that may overlap on the GPU -- on different streams
// without ordering between them -- race on the array and must not be issued.
// Limits: requests whose workspace (dsa_indexer_topk_workspace_size) exceeds the array are
// rejected with DSA_ERR_WORKSPACE. No cudaMalloc, cudaFree or allocating library call is made.
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "status.cuh"

namespace {

constexpr size_t kScratchBytes = DSA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

}  // namespace

#define DSA_EXPORT __attribute__((visibility("default")))

extern "C" DSA_EXPORT int dsa_indexer_topk_noalloc(
    const void* q_idx, const float* w, const void* k_idx, int64_t n_kv_rows, const int32_t* cu,
    int n_req, const int32_t* pos, const int32_t* bid, int64_t n_q, int Hi, int Di, int k,
    int max_ctx, const int32_t* block_table, int max_pages, int page_size, int32_t* topk,
    dsa_stream_t stream) {
  if (n_q < 0 || max_ctx < 1 || k < 1)
    return dsa::fail(DSA_ERR_INVALID, "indexer_topk_noalloc: need n_q >= 0, max_ctx >= 1, k >= 1");
  const size_t need = dsa_indexer_topk_workspace_size(n_q, max_ctx, k);
  if (need > kScratchBytes)
    return dsa::fail(DSA_ERR_WORKSPACE,
                     "indexer_topk_noalloc: n_q=%lld, max_ctx=%d need %zu bytes of scratch, more "
                     "than the %zu-byte static array; use dsa_indexer_topk with a caller buffer",
                     static_cast<long long>(n_q), max_ctx, need, kScratchBytes);
  int dev = 0;
  DSA_CHECK_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices)
    return dsa::fail(DSA_ERR_UNSUPPORTED, "indexer_topk_noalloc: device %d beyond %d", dev,
                     kMaxDevices);
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess) return dsa::cuda_fail(e, "cudaGetSymbolAddress(scratch)");
      g_scratch_ptr[dev] = p;
    }
    scratch = g_scratch_ptr[dev];
  }
  return dsa_indexer_topk(q_idx, w, k_idx, n_kv_rows, cu, n_req, pos, bid, n_q, Hi, Di, k, max_ctx,
                          block_table, max_pages, page_size, topk, scratch, kScratchBytes, stream);
}
