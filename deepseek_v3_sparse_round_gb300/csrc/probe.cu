// Row-gather throughput probe: the two ways the sparse MLA could bring its selected latent rows
// (576 bf16 = 1,152 B each) into shared memory, timed on their own with nothing consuming the
// tiles. Each CTA fills a 3-slot ring of 48-row tiles in the MLA's layout (nine 128B-swizzled
// 64-column atoms per tile) from a list of row indices, and a consumer lane hands every slot
// back as soon as it is full, so only the gather's own rate and latency bound the loop.
//
//   mode 0 (the MLA's path): three warps per slot, 16-byte cp.async copies, one lane per 16-byte
//     chunk of a row; each warp waits for its copies, fences them for the async proxy and
//     arrives on the slot's full barrier.
//   mode 1: TMA tile::gather4 (four rows of one 64-column box per instruction, 108 per tile),
//     issued by `issuers` lanes of one warp, completing on the slot's full barrier by bytes.
//   mode 2: both at once: atoms 0-7 by mode 0's cp.async warps, atom 8 (the rope columns) by
//     12 tile::gather4 issued by lane 0 of the slot's first gather warp.
//   mode 4: as mode 0 through registers: 16-byte ld.global (L1 no-allocate) and st.shared,
//     each warp keeping two rows' nine chunks in flight per lane.
//   mode 5: both paths at once: atoms 0-4 of every row through registers as in mode 4,
//     atoms 5-8 by cp.async as in mode 0.
//   mode 6: as mode 4 with all four of a warp's row groups in flight at once.
//   mode 7: not a gather: each tile is the 48 consecutive rows starting at its first listed row,
//     loaded as nine 64-column x 48-row TMA boxes (128B swizzle) by one lane (the rate for a
//     run of consecutive keys, e.g. every key of a short history).
//   mode 3: not a gather: the rate of the DSMEM path between the two CTAs of a cluster (what
//     the MLA's courier uses). Each CTA pushes 192 KB per round into its peer's shared memory
//     with six 32 KB bulk copies that complete on the peer's barrier; a cluster barrier keeps
//     the two CTAs in step; n_tiles rounds.
//
// Every wait is bounded; row indices outside [0, n_rows) are replaced by row 0 and reported as
// DSA_DEVERR_BAD_INDEX. Each CTA writes the clock cycles its loop took.
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "status.cuh"
#include "tmap.cuh"

namespace dsa {
namespace {

constexpr int kRows = 48, kAtoms = 9, kAtomBytes = kRows * 128, kTile = kAtoms * kAtomBytes;
constexpr int kSlots = 3, kWarpsPerSlot = 3, kGatherWarps = kSlots * kWarpsPerSlot;
constexpr int kThreads = 32 * (kGatherWarps + 1);           // + the consumer warp
constexpr int kSmem = kSlots * kTile;                       // 162 KB, 1 KB aligned tiles
constexpr uint32_t kSite = 0xF0u;
constexpr long long kLimit = 2000000000ll;                  // about a second per wait


// Register path of the gather (modes 4-6): this warp's row groups (part, part + 3, ...),
// kInFlight at a time, atoms 0..kReg-1 by 16-byte ld.global + st.shared, the rest (if any) by
// cp.async issued first.
template <int kInFlight, int kReg, typename RowAt, typename FullBar, typename EmptyBar>
__device__ __forceinline__ void reg_gather(const __nv_bfloat16* __restrict__ c, uint32_t sbase,
                                           uint8_t* smem, uint32_t warp, uint32_t lane,
                                           int n_tiles, RowAt& row_at, FullBar& full,
                                           EmptyBar& empty, uint32_t* abort_flag) {
  const int s = static_cast<int>(warp) % kSlots, part = static_cast<int>(warp) / kSlots;
  const int chunk = static_cast<int>(lane & 7);
  constexpr int kGroups = kRows / 4 / kWarpsPerSlot;        // 4 row groups of 4 rows per warp
  static_assert(kGroups % kInFlight == 0, "row groups in flight");
  for (int j = s; j < n_tiles; j += kSlots) {
    if (!warp_wait(empty(s), static_cast<uint32_t>(((j / kSlots) & 1) ^ 1), kSite | 4u, abort_flag, kLimit)) break;
    if (kReg < kAtoms) {
      for (int i = part; i < kRows / 4; i += kWarpsPerSlot) {
        const int r = static_cast<int>(lane >> 3) + 4 * i;
        const __nv_bfloat16* src = c + static_cast<int64_t>(row_at(j, r)) * (kAtoms * 64) + chunk * 8;
        const uint32_t dst = sbase + s * kTile + r * 128 + ((chunk ^ (r & 7)) * 16);
        for (int a = kReg; a < kAtoms; ++a) cp_async16(dst + a * kAtomBytes, src + a * 64, 16u);
      }
      cp_async_commit();
    }
#pragma unroll
    for (int i0 = 0; i0 < kGroups; i0 += kInFlight) {
      uint4 v[kInFlight][kReg];
#pragma unroll
      for (int u = 0; u < kInFlight; ++u) {
        const int r = static_cast<int>(lane >> 3) + 4 * (part + kWarpsPerSlot * (i0 + u));
        const uint4* src = reinterpret_cast<const uint4*>(
            c + static_cast<int64_t>(row_at(j, r)) * (kAtoms * 64) + chunk * 8);
#pragma unroll
        for (int a = 0; a < kReg; ++a) v[u][a] = ld_nc_v4(src + a * 8);
      }
#pragma unroll
      for (int u = 0; u < kInFlight; ++u) {
        const int r = static_cast<int>(lane >> 3) + 4 * (part + kWarpsPerSlot * (i0 + u));
        uint4* dst = reinterpret_cast<uint4*>(smem + s * kTile + r * 128 + ((chunk ^ (r & 7)) * 16));
#pragma unroll
        for (int a = 0; a < kReg; ++a) dst[a * (kAtomBytes / 16)] = v[u][a];
      }
    }
    if (kReg < kAtoms) cp_async_wait_all();
    fence_proxy_async_smem();
    mbar_arrive(full(s));
  }
  cp_async_wait_all();
}

__global__ void __launch_bounds__(kThreads, 1)
row_gather_probe_kernel(const __grid_constant__ CUtensorMap tm, const __nv_bfloat16* __restrict__ c,
                        int64_t n_rows, const int32_t* __restrict__ rows, int n_tiles, int mode,
                        int issuers, unsigned long long* __restrict__ cycles) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[2 * kSlots];
  __shared__ uint32_t abort_flag;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t warp = warp_id(), lane = lane_id();
  auto full = [&](int s) { return smem_u32(&bars[s]); };
  auto empty = [&](int s) { return smem_u32(&bars[kSlots + s]); };
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSlots; ++s) {
      // modes 1 and 7: one arrival with the byte count; the others: every gather lane
      mbar_init(full(s), mode == 1 || mode == 7 ? 1 : 32 * kWarpsPerSlot);
      mbar_init(empty(s), 1);
    }
    abort_flag = (sbase & 1023u) == 0 ? 0u : 1u;
    if (abort_flag) report_device_error(kErrBadIndex | kSite | 0xFu);   // ring not 1 KB aligned
    fence_mbar_init();
  }
  __syncthreads();
  const int32_t* my_rows = rows + static_cast<int64_t>(blockIdx.x) * n_tiles * kRows;
  bool bad = false;
  auto row_at = [&](int j, int r) {
    const int32_t v = __ldg(my_rows + static_cast<int64_t>(j) * kRows + r);
    if (v < 0 || v >= n_rows) { bad = true; return 0; }
    return static_cast<int>(v);
  };
  const long long t0 = clock64();
  if (warp == kGatherWarps) {
    // consumer: every full slot goes straight back
    for (int j = 0; j < n_tiles; ++j) {
      const int s = j % kSlots;
      if (!warp_wait(full(s), static_cast<uint32_t>((j / kSlots) & 1), kSite, &abort_flag, kLimit)) break;
      if (lane == 0) mbar_arrive(empty(s));
    }
  } else if (mode == 0 || mode == 2) {
    const int s = static_cast<int>(warp) % kSlots, part = static_cast<int>(warp) / kSlots;
    const int chunk = static_cast<int>(lane & 7);
    const uint32_t stage = sbase + s * kTile;
    const int n_cp = mode == 0 ? kAtoms : kAtoms - 1;       // atoms copied by cp.async
    int last = -1;                                   // mode 2: the last tile this lane's TMA filled
    for (int j = s; j < n_tiles; j += kSlots) {
      if (!warp_wait(empty(s), static_cast<uint32_t>(((j / kSlots) & 1) ^ 1), kSite | 1u, &abort_flag, kLimit)) break;
      if (mode == 2 && part == 0 && lane == 0) {
        // atom 8 by TMA: its bytes complete on the slot's full barrier (the count is added
        // without an arrival of its own, before this lane's arrival below)
        mbar_add_tx(full(s), kAtomBytes);
        for (int q4 = 0; q4 < kRows / 4; ++q4)
          tma_gather4(stage + (kAtoms - 1) * kAtomBytes + q4 * 4 * 128, &tm, (kAtoms - 1) * 64,
                      row_at(j, 4 * q4), row_at(j, 4 * q4 + 1), row_at(j, 4 * q4 + 2),
                      row_at(j, 4 * q4 + 3), full(s));
        last = j;
      }
      for (int i = part; i < kRows / 4; i += kWarpsPerSlot) {
        const int r = static_cast<int>(lane >> 3) + 4 * i;
        const __nv_bfloat16* src = c + static_cast<int64_t>(row_at(j, r)) * (kAtoms * 64) + chunk * 8;
        const uint32_t dst = stage + r * 128 + ((chunk ^ (r & 7)) * 16);
        for (int a = 0; a < n_cp; ++a) cp_async16(dst + a * kAtomBytes, src + a * 64, 16u);
      }
      cp_async_commit();
      cp_async_wait_all();
      fence_proxy_async_smem();
      mbar_arrive(full(s));
    }
    cp_async_wait_all();
    if (last >= 0) {
      // unwinding: let this lane's last TMA fill land before the CTA can exit (bounded)
      const long long w0 = clock64();
      while (!mbar_try_wait(full(s), static_cast<uint32_t>((last / kSlots) & 1)) &&
             clock64() - w0 < kLimit) {
      }
    }
  } else if (mode == 4) {
    reg_gather<2, kAtoms>(c, sbase, smem, warp, lane, n_tiles, row_at, full, empty, &abort_flag);
  } else if (mode == 5) {
    reg_gather<2, 5>(c, sbase, smem, warp, lane, n_tiles, row_at, full, empty, &abort_flag);
  } else if (mode == 6) {
    reg_gather<4, kAtoms>(c, sbase, smem, warp, lane, n_tiles, row_at, full, empty, &abort_flag);
  } else if (warp == 0) {
    int last = -1;                                   // the last tile this warp started
    for (int j = 0; j < n_tiles; ++j) {
      const int s = j % kSlots;
      if (!warp_wait(empty(s), static_cast<uint32_t>(((j / kSlots) & 1) ^ 1), kSite | 2u, &abort_flag, kLimit)) break;
      if (lane == 0) mbar_expect_tx(full(s), kTile);
      __syncwarp();
      if (mode == 7) {
        if (lane == 0) {
          // rows past the end of the cache read the fill value (zero); the start is in range
          const int r0 = row_at(j, 0);
          for (int a = 0; a < kAtoms; ++a)
            tma_load_2d(sbase + s * kTile + a * kAtomBytes, &tm, a * 64, r0, full(s));
        }
      } else if (static_cast<int>(lane) < issuers) {
        for (int g = static_cast<int>(lane); g < kAtoms * (kRows / 4); g += issuers) {
          const int a = g / (kRows / 4), q4 = g % (kRows / 4);
          tma_gather4(sbase + s * kTile + a * kAtomBytes + q4 * 4 * 128, &tm, a * 64,
                      row_at(j, 4 * q4), row_at(j, 4 * q4 + 1), row_at(j, 4 * q4 + 2),
                      row_at(j, 4 * q4 + 3), full(s));
        }
      }
      __syncwarp();
      last = j;
    }
    // unwinding: let the loads already issued land before the CTA can exit (bounded)
    for (int j = last - kSlots + 1; j <= last; ++j) {
      if (j < 0) continue;
      const long long w0 = clock64();
      while (!mbar_try_wait(full(j % kSlots), static_cast<uint32_t>((j / kSlots) & 1)) &&
             clock64() - w0 < kLimit) {
      }
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) report_device_error(kErrBadIndex | kSite);
  __syncthreads();
  if (threadIdx.x == 0) cycles[blockIdx.x] = static_cast<unsigned long long>(clock64() - t0);
}

constexpr int kXChunk = 32768, kXChunks = 6, kXRound = kXChunk * kXChunks;   // 192 KB a round

__global__ void __launch_bounds__(128, 1)
dsmem_probe_kernel(int rounds, unsigned long long* __restrict__ cycles) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  const uint32_t sbase = smem_u32(smem), b = smem_u32(&bar);
  const uint32_t peer = cluster_ctarank() ^ 1u;
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    abort_flag = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  cluster_sync();                                    // the peer's barrier exists from here on
  const long long t0 = clock64();
  // Every CTA runs every round (no early exit), so both reach every cluster barrier; a wait
  // that gives up only sets the error word and the abort flag (later waits return at once).
  for (int r = 0; r < rounds; ++r) {
    if (threadIdx.x == 0) mbar_expect_tx(b, kXRound);   // this round's incoming bytes
    cluster_sync();                                  // both CTAs armed before any copy lands
    if (threadIdx.x == 0) {
      // the source is the CTA's own buffer while the peer's copies land in it: the bytes are
      // not used, only their rate
      for (int i = 0; i < kXChunks; ++i)
        bulk_copy_to_peer(sbase + i * kXChunk, sbase + i * kXChunk, kXChunk, b, peer);
      bulk_commit();
      mbar_wait(b, static_cast<uint32_t>(r & 1), kSite | 3u, &abort_flag, kLimit);
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    bulk_wait_all();                                 // this CTA's outgoing copies are done
    cycles[blockIdx.x] = static_cast<unsigned long long>(clock64() - t0);
  }
  __syncthreads();
  cluster_sync();                                    // no CTA leaves while its peer may write
}

}  // namespace

int probe_row_gather(const void* c, int64_t n_rows, const int32_t* rows, int n_ctas, int n_tiles,
                     int mode, int issuers, unsigned long long* cycles, cudaStream_t stream) {
  if (mode == 3) {
    DSA_CHECK_CUDA(cudaFuncSetAttribute(dsmem_probe_kernel,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, kXRound));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(n_ctas));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = kXRound;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    DSA_CHECK_CUDA(cudaLaunchKernelEx(&cfg, dsmem_probe_kernel, n_tiles, cycles));
    return DSA_OK;
  }
  CUtensorMap tm;
  // one-row boxes for tile::gather4, 48-row boxes for the runs of mode 7
  int rc = make_tmap_bf16_2d(&tm, c, static_cast<uint64_t>(n_rows), kAtoms * 64, kAtoms * 128,
                             64, mode == 7 ? kRows : 1, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  DSA_CHECK_CUDA(cudaFuncSetAttribute(row_gather_probe_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem));
  row_gather_probe_kernel<<<n_ctas, kThreads, kSmem, stream>>>(
      tm, static_cast<const __nv_bfloat16*>(c), n_rows, rows, n_tiles, mode, issuers, cycles);
  DSA_CHECK_CUDA(cudaGetLastError());
  return DSA_OK;
}

cudaError_t probe_read_errors(uint32_t* flags) { return read_and_clear_device_error(flags); }

}  // namespace dsa
