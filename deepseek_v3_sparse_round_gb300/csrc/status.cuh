// Status codes, the per-translation-unit device error word, and host-side error text.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/dsa_rr.h"

namespace dsa {

// Device error word bits (ORed in by kernels; read and cleared by dsa_read_device_errors).
enum : uint32_t {
  kErrTimeout = DSA_DEVERR_TIMEOUT,        // a bounded wait gave up; low byte = wait site
  kErrBadIndex = DSA_DEVERR_BAD_INDEX,     // an input index was out of range and was skipped
  kErrBadLength = DSA_DEVERR_BAD_LENGTH,   // a query row longer than the stated maximum
};

// One word per translation unit (internal linkage: no relocatable device code needed).
static __device__ uint32_t g_device_error;

__device__ __forceinline__ void report_device_error(uint32_t code) {
  atomicOr(&g_device_error, code);
}

// Host: copy this translation unit's word into *out (ORed) and clear it. Synchronous.
static inline cudaError_t read_and_clear_device_error(uint32_t* out) {
  uint32_t v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v));
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
  *out |= v;
  return e;
}

// Host-side error reporting (thread-local message, read by dsa_last_error_string()).
void set_error(const char* fmt, ...);
int fail(int code, const char* fmt, ...);
int cuda_fail(cudaError_t e, const char* what);

}  // namespace dsa

#define DSA_CHECK_CUDA(expr)                                    \
  do {                                                          \
    cudaError_t _e = (expr);                                    \
    if (_e != cudaSuccess) return ::dsa::cuda_fail(_e, #expr);  \
  } while (0)
