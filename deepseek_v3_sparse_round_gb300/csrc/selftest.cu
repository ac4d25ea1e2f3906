// Self-test of the bounded in-kernel wait that every tcgen05 kernel of the library uses.
//
// One CTA initialises an mbarrier that nothing ever arrives on and waits for its first phase
// with the library's bounded wait (the same mbar_wait the indexer and MLA kernels use), given a
// short limit. The wait gives up after the limit, sets DSA_DEVERR_TIMEOUT with site 0xEE in the
// device error word and the kernel returns normally: nothing faults or hangs, and the host reads
// the status with dsa_read_device_errors. No other memory is touched and no asynchronous copy
// or tensor-core operation is in flight when the kernel exits.
#include <cstdint>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "status.cuh"

namespace dsa {
namespace {

constexpr uint32_t kSiteSelftest = 0xEEu;

__global__ void __launch_bounds__(32) bounded_wait_selftest_kernel(long long limit_cycles) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    abort_flag = 0u;
    fence_mbar_init();
  }
  __syncwarp();
  // The barrier's phase 0 never completes: only the time limit ends this wait.
  const bool ok = warp_wait(b, 0u, kSiteSelftest, &abort_flag, limit_cycles);
  if (ok && threadIdx.x == 0) report_device_error(kErrBadIndex | kSiteSelftest);  // impossible
}

}  // namespace

int selftest_bounded_wait(long long limit_cycles, cudaStream_t stream) {
  bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_cycles);
  DSA_CHECK_CUDA(cudaGetLastError());
  return DSA_OK;
}

cudaError_t selftest_read_errors(uint32_t* flags) { return read_and_clear_device_error(flags); }

}  // namespace dsa
