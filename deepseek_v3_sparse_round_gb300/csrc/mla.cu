// Sparse MLA on tcgen05 tensor cores: every shard query attends, with all heads at once, to the
// latent rows its top-k selected ("[RFC]: Parallel strategy for Deepseek v3.2 like models":
// "full head on mla part, high tflops").
//
//   S[h, j] = scale * q[t, h, :] . c[row_j, :]          (dqk = 576 = 512 latent + 64 rope)
//   o[t, h, :] = sum_j softmax_j(S[h, :]) c[row_j, 0:dv]  (dv = 512), lse[t, h] = ln sum exp S
//
// Two kernels:
//   * sparse_mla_pair_kernel (H = 128, dqk = 576, dv = 512): a persistent grid of CTA pairs;
//     see the comment above it.
//   * sparse_mla_kernel (small heads, H <= 128 with dv <= 256; built for H = 8, dqk = 80,
//     dv = 64): one CTA per query owns the whole contraction and output. Each 64-key tile:
//     TMA tile::gather4 brings the selected rows into a 4-stage ring; one MMA chain computes S
//     (128 x 64 fp32) in TMEM; the softmax warps run the online softmax (exp2, running
//     maximum, rescaling O only when the maximum grows by more than 2^8), write P as bf16 into
//     a swizzled smem tile and the MMA warp accumulates O += P . V, where V is the same
//     gathered tile read MN-major. QK(j+1) is issued before PV(j) so the tensor pipe works
//     while the softmax of tile j runs.
#include <algorithm>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "status.cuh"
#include "tmap.cuh"

namespace dsa {
namespace {

constexpr int kTileKeys = 64;
constexpr int kMaxK = 4096;
constexpr int kPageRows = 64;

template <int H, int DQK, int DV>
struct MlaShape {
  static constexpr int kGAtoms = (DQK + 63) / 64;            // 64-column swizzle atoms per row
  static constexpr int kQKSteps = DQK / 16;                  // k-steps (16 dims)
  static constexpr int kQCols = ((DQK / 2) + 15) / 16 * 16;  // TMEM columns for Q
  static constexpr int kDVc = DV;                            // output dims (one CTA)
  static constexpr int kAtomBytes = kTileKeys * 128;         // 64 rows x 128 B
  static constexpr int kStageBytes = kGAtoms * kAtomBytes;
  static constexpr int kStages = 4;
  static constexpr int kPBytes = 128 * 128;                  // 128 rows x 64 keys bf16
  static constexpr int kOffKV = 0;
  static constexpr int kOffP = kStages * kStageBytes;
  static constexpr int kOffMask = kOffP + 2 * kPBytes;
  static constexpr int kOffBar = kOffMask + (kMaxK / kTileKeys) * 8;
  static constexpr int kNumBars = 2 * kStages + 12;
  static constexpr int kOffTmem = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffTmem + 4;
  static constexpr int kOffNTiles = kOffAbort + 4;
  static constexpr int kSmem = kOffNTiles + 8;
  // TMEM columns: O | S | Q
  static constexpr int kColO = 0;
  static constexpr int kColS = kDVc < 64 ? 64 : kDVc;
  static constexpr int kColQ = kColS + kTileKeys;
  static constexpr int kTmemCols = (kColQ + kQCols) <= 256 ? 256 : 512;
  static constexpr int kThreads = 192;                       // 4 softmax warps + TMA + MMA
  static_assert(H <= 128, "heads per CTA");
  static_assert(DQK % 16 == 0, "qk k-steps");
  static_assert(kColQ + kQCols <= 512, "TMEM budget");
  static_assert(kSmem <= 232448, "smem budget");
  static_assert(kDVc % 16 == 0 && kDVc <= 256, "PV N: one CTA holds O");
};

struct KvMap {
  const int32_t* cu;           // contiguous mode
  const int32_t* block_table;  // paged mode (nullptr: contiguous)
  int max_pages;
  int n_req;
  int64_t n_rows;
  const int32_t* pos;          // query positions (nullptr: not given)
};

// Largest top-k entry query t of request b may hold: the last position of its request
// (contiguous), the last position its block-table row can address (paged), and, when the
// positions are given, pos_t (a key after the query is not in its causal history).
__device__ __forceinline__ int entry_limit(const KvMap& m, int b, int64_t t) {
  int lim;
  if (m.block_table == nullptr) {
    lim = __ldg(m.cu + b + 1) - __ldg(m.cu + b) - 1;
  } else {
    const int64_t span = static_cast<int64_t>(m.max_pages) * kPageRows - 1;
    lim = span < 0x7FFFFFFF ? static_cast<int>(span) : 0x7FFFFFFF;
  }
  if (m.pos != nullptr) lim = min(lim, __ldg(m.pos + t));
  return lim;
}

// KV row of position s in request b, or n_rows (read as zeros) when it is not addressable.
// s < 0 is padding; s > lim (past the query or its request) is an invalid index: skipped and
// recorded in *bad.
__device__ __forceinline__ int32_t kv_row(const KvMap& m, int b, int s, int lim, bool* bad) {
  if (s < 0) return static_cast<int32_t>(m.n_rows);
  if (s > lim) { *bad = true; return static_cast<int32_t>(m.n_rows); }
  int64_t r;
  if (m.block_table == nullptr) {
    r = static_cast<int64_t>(__ldg(m.cu + b)) + s;
  } else {
    const int pi = s / kPageRows;
    const int page = pi < m.max_pages ? __ldg(m.block_table + static_cast<int64_t>(b) * m.max_pages + pi) : -1;
    r = page < 0 ? m.n_rows : static_cast<int64_t>(page) * kPageRows + s % kPageRows;
  }
  if (r < 0 || r >= m.n_rows) { *bad = true; return static_cast<int32_t>(m.n_rows); }
  return static_cast<int32_t>(r);
}

template <int H, int DQK, int DV>
__global__ void __launch_bounds__(MlaShape<H, DQK, DV>::kThreads, 1)
sparse_mla_kernel(const __grid_constant__ CUtensorMap tm_c, const __nv_bfloat16* __restrict__ q,
                  const int32_t* __restrict__ bid, const int32_t* __restrict__ topk, int k,
                  KvMap kv, float scale_log2, __nv_bfloat16* __restrict__ o,
                  float* __restrict__ lse) {
  using S = MlaShape<H, DQK, DV>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const uint32_t warp = warp_id(), lane = lane_id();
  const int64_t t = blockIdx.x;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + S::kOffAbort);
  uint64_t* masks = reinterpret_cast<uint64_t*>(smem + S::kOffMask);
  auto bar = [&](int i) { return sbase + S::kOffBar + 8u * static_cast<uint32_t>(i); };
  const int kKvFull = 0, kKvEmpty = S::kStages, kQReady = 2 * S::kStages, kSFull = kQReady + 1,
            kSEmpty = kQReady + 2, kPFull = kQReady + 3, kPEmpty = kQReady + 5,
            kOReady = kQReady + 7, kOFinal = kQReady + 8;

  const bool aligned = (sbase & 1023u) == 0;
  if (threadIdx.x == 0) {
    for (int i = 0; i < S::kStages; ++i) { mbar_init(bar(kKvFull + i), 1); mbar_init(bar(kKvEmpty + i), 1); }
    mbar_init(bar(kQReady), 128);
    mbar_init(bar(kSFull), 1);
    mbar_init(bar(kSEmpty), 4);
    for (int i = 0; i < 2; ++i) { mbar_init(bar(kPFull + i), 128); mbar_init(bar(kPEmpty + i), 1); }
    mbar_init(bar(kOReady), 1);
    mbar_init(bar(kOFinal), 1);
    *abort_flag = aligned ? 0u : 1u;
    if (!aligned) report_device_error(kErrBadIndex | 0xB1u);
    fence_mbar_init();
  }
  // Tile validity masks and the number of tiles up to the last valid entry.
  const int32_t* trow = topk + t * k;
  const int n_tiles_max = (k + kTileKeys - 1) / kTileKeys;
  const int b = __ldg(bid + t);
  const bool b_ok = b >= 0 && b < kv.n_req;
  const int lim = b_ok ? entry_limit(kv, b, t) : -1;
  if (threadIdx.x == 0) *reinterpret_cast<volatile int*>(smem + S::kOffNTiles) = 0;
  __syncthreads();
  for (int tile = static_cast<int>(warp); tile < n_tiles_max; tile += S::kThreads / 32) {
    const int j0 = tile * kTileKeys + static_cast<int>(lane), j1 = j0 + 32;
    const int e0 = j0 < k ? __ldg(trow + j0) : -1, e1 = j1 < k ? __ldg(trow + j1) : -1;
    const bool v0 = e0 >= 0 && e0 <= lim;
    const bool v1 = e1 >= 0 && e1 <= lim;
    const uint32_t b0 = __ballot_sync(0xffffffffu, v0), b1 = __ballot_sync(0xffffffffu, v1);
    if (lane == 0) {
      masks[tile] = static_cast<uint64_t>(b0) | (static_cast<uint64_t>(b1) << 32);
      if (b0 | b1) atomicMax(reinterpret_cast<int*>(smem + S::kOffNTiles), tile + 1);
    }
  }
  if (warp == 0) tmem_alloc<S::kTmemCols>(sbase + S::kOffTmem);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + S::kOffTmem);
  const int n_tiles = *reinterpret_cast<volatile int*>(smem + S::kOffNTiles);

  if (warp == 4) {
    // ------------------------------------------------------------------ TMA gather producer
    if (lane == 0) tma_prefetch_desc(&tm_c);
    bool bad = !b_ok;
    int stage = 0, issued = 0;
    uint32_t phase = 0;
    for (int j = 0; j < n_tiles; ++j) {
      bool ok = true;
      if (lane == 0) ok = mbar_wait(bar(kKvEmpty + stage), phase ^ 1u, 0x11, abort_flag);
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
      if (lane == 0) mbar_expect_tx(bar(kKvFull + stage), S::kStageBytes);
      __syncwarp();
      if (lane < kTileKeys / 4) {
        int32_t rows[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int e = j * kTileKeys + static_cast<int>(lane) * 4 + i;
          const int s = (e < k && b_ok) ? __ldg(trow + e) : -1;
          rows[i] = kv_row(kv, b_ok ? b : 0, s, lim, &bad);
        }
        const uint32_t dst = sbase + S::kOffKV + stage * S::kStageBytes + lane * 4 * 128;
#pragma unroll
        for (int a = 0; a < S::kGAtoms; ++a)
          tma_gather4(dst + a * S::kAtomBytes, &tm_c, a * 64, rows[0], rows[1], rows[2], rows[3],
                      bar(kKvFull + stage));
      }
      ++issued;
      if (++stage == S::kStages) { stage = 0; phase ^= 1u; }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) report_device_error(kErrBadIndex);
    if (*abort_flag && lane == 0) {                   // let issued copies land before exiting
      for (int i = 0; i < S::kStages && i < issued; ++i) {
        const int jl = issued - 1 - i;
        const long long t0 = clock64();
        while (!mbar_try_wait(bar(kKvFull + jl % S::kStages), (jl / S::kStages) & 1u) &&
               clock64() - t0 < kWaitLimitCycles) {
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = idesc_bf16(128, kTileKeys, 0, 0);
      const uint32_t idesc_pv = idesc_bf16(128, S::kDVc, 0, 1);
      auto pv = [&](int j) -> bool {
        if (!mbar_wait(bar(kPFull + (j & 1)), (j >> 1) & 1, 0x12, abort_flag)) return false;
        tc_fence_after();
        const int st = j % S::kStages;
        const uint32_t p_base = sbase + S::kOffP + (j & 1) * S::kPBytes;
        const uint32_t v_base = sbase + S::kOffKV + st * S::kStageBytes;
#pragma unroll
        for (int kk = 0; kk < kTileKeys / 16; ++kk) {
          const uint64_t da = smem_desc(p_base + kk * 32, 16, 1024, kSwizzle128B);
          const uint64_t dv = smem_desc(v_base + kk * 2048, S::kAtomBytes, 1024, kSwizzle128B);
          umma_ss(tmem + S::kColO, da, dv, idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(bar(kPEmpty + (j & 1)));
        umma_commit(bar(kKvEmpty + st));
        umma_commit(bar(kOReady));
        return true;
      };
      bool ok = mbar_wait(bar(kQReady), 0, 0x13, abort_flag);
      tc_fence_after();
      for (int j = 0; j < n_tiles && ok; ++j) {
        const int st = j % S::kStages;
        if (!mbar_wait(bar(kKvFull + st), (j / S::kStages) & 1, 0x14, abort_flag)) { ok = false; break; }
        if (!mbar_wait(bar(kSEmpty), (j & 1) ^ 1, 0x15, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t kv_base = sbase + S::kOffKV + st * S::kStageBytes;
#pragma unroll
        for (int kk = 0; kk < S::kQKSteps; ++kk) {
          const int a = kk / 4, off = (kk % 4) * 32;
          const uint64_t db = smem_desc(kv_base + a * S::kAtomBytes + off, 16, 1024, kSwizzle128B);
          umma_ts(tmem + S::kColS, tmem + S::kColQ + kk * 8, db, idesc_qk, kk > 0 ? 1u : 0u);
        }
        umma_commit(bar(kSFull));
        if (j > 0 && !pv(j - 1)) { ok = false; break; }
      }
      if (ok && n_tiles > 0 && pv(n_tiles - 1)) umma_commit(bar(kOFinal));
    }
  } else {
    // ------------------------------------------------------------------ softmax + epilogue
    const int h = static_cast<int>(threadIdx.x);     // head row == TMEM lane
    const uint32_t lane_base = (warp * 32u) << 16;
    // Q slice -> TMEM (A operand of QK).
    {
      const uint4* src = reinterpret_cast<const uint4*>(q + (t * H + (h < H ? h : 0)) * DQK);
#pragma unroll
      for (int c0 = 0; c0 < S::kQCols; c0 += 16) {
        uint32_t r[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int e = (c0 + 4 * i) * 2;              // first element of this 16-byte chunk
          uint4 v = make_uint4(0, 0, 0, 0);
          if (h < H && e < DQK) v = __ldg(src + e / 8);
          r[4 * i] = v.x; r[4 * i + 1] = v.y; r[4 * i + 2] = v.z; r[4 * i + 3] = v.w;
        }
        tmem_st16(tmem + lane_base + S::kColQ + c0, r);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(kQReady));
    }
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      if (!warp_wait(bar(kSFull), j & 1, 0x16, abort_flag)) { ok = false; break; }
      tc_fence_after();
      float sv[kTileKeys];
      {
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + S::kColS, r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) sv[i] = __uint_as_float(r[i]);
        tmem_ld32(tmem + lane_base + S::kColS + 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) sv[32 + i] = __uint_as_float(r[i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kSEmpty));
      // online softmax in the log2 domain
      const uint64_t mk = masks[j];
      float mt = -INFINITY;
#pragma unroll
      for (int i = 0; i < kTileKeys; ++i) {
        sv[i] = ((mk >> i) & 1ull) ? sv[i] * scale_log2 : -INFINITY;
        mt = fmaxf(mt, sv[i]);
      }
      float alpha = 1.f;
      if (m_run == -INFINITY) {
        m_run = mt;                                    // first tile with a valid key (or still -inf)
      } else if (mt > m_run + 8.f) {
        alpha = ex2_approx(m_run - mt);
        m_run = mt;
      }
      // Rescale this row of O when its reference maximum moved (rare): after PV(j-1) finished.
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
        if (!warp_wait(bar(kOReady), (j - 1) & 1, 0x19, abort_flag)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < S::kDVc; c0 += 16) {
          uint32_t r[16];
          tmem_ld16(tmem + lane_base + S::kColO + c0, r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tmem_st16(tmem + lane_base + S::kColO + c0, r);
        }
        tmem_wait_st();
      }
      l_run *= alpha;
      float psum = 0.f;
      uint32_t pk[kTileKeys / 2];
#pragma unroll
      for (int i = 0; i < kTileKeys; i += 2) {
        const float p0 = m_run == -INFINITY ? 0.f : ex2_approx(sv[i] - m_run);
        const float p1 = m_run == -INFINITY ? 0.f : ex2_approx(sv[i + 1] - m_run);
        psum += p0 + p1;
        pk[i / 2] = bf16x2_bits(p0, p1);
      }
      l_run += psum;
      // P row -> swizzled K-major smem tile (A operand of PV)
      if (!warp_wait(bar(kPEmpty + (j & 1)), ((j >> 1) & 1) ^ 1, 0x1A, abort_flag)) { ok = false; break; }
      uint8_t* prow = smem + S::kOffP + (j & 1) * S::kPBytes + (h >> 3) * 1024 + (h & 7) * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(prow + ((c ^ (h & 7)) * 16)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(kPFull + (j & 1)));
    }
    // epilogue: O / l -> bf16, lse
    if (ok && n_tiles > 0) ok = warp_wait(bar(kOFinal), 0, 0x1B, abort_flag);
    tc_fence_after();
    const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll 1
    for (int c0 = 0; c0 < S::kDVc; c0 += 16) {
      uint32_t r[16];
      if (ok && n_tiles > 0) {
        tmem_ld16(tmem + lane_base + S::kColO + c0, r);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] = 0u;
      }
      if (h < H) {
        uint32_t pk[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          pk[i] = bf16x2_bits(__uint_as_float(r[2 * i]) * inv_l, __uint_as_float(r[2 * i + 1]) * inv_l);
        uint4* dst = reinterpret_cast<uint4*>(o + (t * H + h) * DV + c0);
        dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      }
    }
    if (lse != nullptr && h < H)
      lse[t * H + h] = l_run > 0.f ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
  }

  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc<S::kTmemCols>(tmem);
  }
}

// =============================================================================================
// H = 128, dqk = 576, dv = 512: a cluster of two CTAs per query with split roles.
//   CTA 0 ("S side"): Q (128 x 576 bf16) in TMEM as the A operand (288 columns) and one S tile
//     of 128 x 48 fp32 per ring slot, so QK(j+1) runs while the softmax of tile j runs. One
//     warp-uniform QK issuer takes every tile in order, so it sees every phase of the barriers
//     it waits on (an issuer skipping another issuer's tiles on a 3-slot ring could take a
//     parity two phases ahead). Its softmax warps stage P (bf16), the per-row rescale factors
//     and flags in one of kPBuf staging buffers; a courier warp ships each to CTA 1 with bulk
//     DSMEM copies (one bulk copy moves a tile far faster than per-thread DSMEM stores). A ring
//     slot is free as soon as its QK MMAs finish.
//   CTA 1 ("O side"): O (128 x 512 fp32) fills its TMEM; it accumulates O += P . V with two
//     N = 256 MMAs per 16 keys and writes o = O / l at the end (TMA stores).
// Each CTA gathers the selected rows it needs into its own 3-slot ring of 48-key tiles (CTA 0:
// all 576 columns, CTA 1: the 512 latent columns), three gather warps per slot. Ahead of a
// query's tiles, CTA 0's ring carries its Q in three TMA-loaded pieces that the QK issuer copies
// into TMEM (tcgen05.cp) once the previous query's QK MMAs are done. The running maximum is
// lazy: O is rescaled only when a row's maximum grows by more than 2^16 (rare; then CTA 1's
// four row warps rescale O between two PV steps).
namespace pair {
constexpr int kH = 128, kDQK = 576, kDV = 512;
constexpr int kKeys = 48;                       // keys per tile
constexpr int kStages = 3;
// validity bits of one query's top-k entries, up to the end of its last tile (+1 word so the
// two-word read of a tile's bits stays inside the buffer)
constexpr int kMaskWords = ((kMaxK + kKeys - 1) / kKeys * kKeys + 31) / 32 + 1;
constexpr int kAtomBytes = kKeys * 128;         // one 64-column swizzle atom of a tile: 6 KB
constexpr int kAtomsS = 9;                      // CTA 0: dims 0..575
constexpr int kAtomsO = 8;                      // CTA 1: dims 0..511
constexpr int kStageS = kAtomsS * kAtomBytes;   // 54 KB
constexpr int kStageO = kAtomsO * kAtomBytes;   // 48 KB
// P (128 rows x 48 keys bf16) in the 32B-swizzled K-major layout: three 16-key atoms of
// 128 rows x 32 B (4 KB each); row h at (h / 8) * 256 + (h % 8) * 32, its 16-byte chunk c at
// (c ^ ((h / 4) % 2)) * 16. 12 KB, all of it used (a 128B-swizzled tile would need 16 KB).
constexpr int kPAtomBytes = 128 * 32;
constexpr int kPBytes = (kKeys / 16) * kPAtomBytes;
constexpr int kAFBytes = 128 * 4 + 16;          // alpha[128] fp32 + flags[4] u32 (528 bytes)
constexpr int kAFStride = 544;
constexpr int kPBuf = 3;                        // P tiles in flight between the CTAs
constexpr int kOffP = kStages * kStageO;        // CTA 1: kPBuf P buffers
constexpr int kPSStride = (kPBytes + kAFBytes + 1023) / 1024 * 1024;  // CTA 0: P + alpha + flags
constexpr int kOffPS = kStages * kStageS;       // CTA 0: kPBuf P staging buffers
constexpr int kOffMask = kOffPS + kPBuf * kPSStride;  // CTA 0: u32 [2][kMaskWords]
constexpr int kEndS = kOffMask + 2 * kMaskWords * 4, kEndO = kOffP + kPBuf * kPBytes;
constexpr int kRegion = ((kEndS > kEndO ? kEndS : kEndO) + 15) / 16 * 16;
// 32 rows x 128 B per row warp, 1 KB aligned (128B swizzle): CTA 1 stages bf16 o in it for
// TMA stores.
constexpr int kOffX = (kRegion + 1023) / 1024 * 1024;
constexpr int kXBytes = 4 * 32 * 128;
constexpr int kOffXO1 = kEndO;                  // CTA 1: second o staging tile per row warp
constexpr int kOffAlpha = kOffX + kXBytes;      // CTA 1: [kPBuf][kAFStride] alpha + flags
constexpr int kOffL = kOffAlpha + kPBuf * kAFStride;  // CTA 1: fp32 [2][128]
constexpr int kOffNT = kOffL + 2 * 128 * 4;     // both: int [2] tiles of the query
constexpr int kOffBar = kOffNT + 8;
constexpr int kNumBars = 4 * kStages + 4 * kPBuf + 13;
constexpr int kOffTmem = kOffBar + kNumBars * 8;
constexpr int kOffAbort = kOffTmem + 4;
constexpr int kOffCorrJ = kOffAbort + 4;
constexpr int kSmem = kOffCorrJ + 4;
constexpr int kColQ = 0, kQCols = kDQK / 2;     // CTA 0 TMEM: Q, then two 64-column S tiles
constexpr int kColS = 288, kSStride = 64;       // S tile of slot s at kColS + 64 s
constexpr int kGatherPerSlot = 3;               // gather warps per ring slot
constexpr int kThreads = 32 * (kGatherPerSlot * kStages + 7);
// warp roles: 0-3 row warps (TMEM lane quadrants); 4 MMA issuer (CTA 0: QK, CTA 1: PV);
// 5..4+kStages and 10.. row gather (warps 5 + s, 10 + s, 13 + s fill ring slot s together);
// 8 the P courier (CTA 0); 9 the query metadata warp (both).
constexpr int kMmaWarp = 4, kGatherWarp0 = 5, kCourierWarp = kGatherWarp0 + kStages,
              kMetaWarp = kCourierWarp + 1, kGatherWarp1 = kMetaWarp + 1;
static_assert(kGatherWarp1 + (kGatherPerSlot - 1) * kStages == kThreads / 32, "warp roles");
constexpr float kLazyLog2 = 16.f;               // rescale O only when the max grows by > 2^16
constexpr float kLazySum = 32768.f;             // 2^(kLazyLog2 - 1): a row sum that checks the max
// CTA 0 brings each query's Q into TMEM through its ring: kQPieces ring entries ahead of the
// query's key tiles, each 128 rows x kQAtomsPerPiece swizzle atoms of 64 dims (128 B per row),
// gathered like key rows and copied into TMEM by the QK issuer (tcgen05.cp).
constexpr int kQPieces = 3, kQAtomsPerPiece = 3;
constexpr int kQAtomBytes = kH * 128;           // 128 rows x 128 B: 16 KB
static_assert(kQPieces * kQAtomsPerPiece * 64 == kDQK, "Q pieces cover the 576 dims");
static_assert(kQAtomsPerPiece * kQAtomBytes <= kStageS, "a Q piece fits a ring slot");
// barrier indices
constexpr int kKvFull = 0, kKvEmpty = kStages, kPStaged = 2 * kStages, kPSEmpty = kPStaged + kPBuf,
              kSFull = kPSEmpty + kPBuf, kSEmpty = kSFull + kStages, kPFull = kSEmpty + kStages,
              kPEmpty = kPFull + kPBuf, kMetaFull = kPEmpty + kPBuf, kMetaEmpty = kMetaFull + 2,
              kLReady = kMetaEmpty + 2, kLEmpty = kLReady + 2, kQFree = kLEmpty + 2,
              kCorrGo = kQFree + 1, kCorrReady = kQFree + 2, kCorrDone = kQFree + 3,
              kOFinal = kQFree + 4;
static_assert(kOFinal + 1 == kNumBars, "barrier count");
static_assert(kSmem <= 232448, "smem budget");
static_assert(kOffPS % 1024 == 0 && kPSStride % 1024 == 0 && kOffP % 1024 == 0 &&
              kPBytes % 1024 == 0, "P tiles: bulk copies 16-byte, swizzle atoms 256-byte aligned");
static_assert(kColS >= kColQ + kQCols && kColS + (kStages - 1) * kSStride + kKeys <= 512,
              "TMEM budget");
static_assert(kAFBytes % 16 == 0, "P staging");
static_assert(kOffXO1 % 1024 == 0 && kOffXO1 + kXBytes <= kRegion, "CTA 1's second o tiles");
static_assert(kKeys == 48, "the gather and softmax split a tile into 32 + 16 entries");
static_assert(kStageS % 1024 == 0 && kStageO % 1024 == 0 && kAtomBytes % 1024 == 0, "SW128");
}  // namespace pair

// Persistent: cluster i of n processes the queries in slots i, i + n, i + 2n, ... of `order` (the
// identity when null). Every role walks the same query sequence and, inside it, the same global
// tile sequence (tiles of earlier queries included), so ring slots, S/P buffers and their
// barrier phases continue across queries.
// Every role waits for every per-query phase in order, also for queries where it has no tile.
__global__ void __launch_bounds__(pair::kThreads, 1)
sparse_mla_pair_kernel(const __grid_constant__ CUtensorMap tm_o,
                       const __grid_constant__ CUtensorMap tm_q,
                       const __nv_bfloat16* __restrict__ c, const __nv_bfloat16* __restrict__ q,
                       const int32_t* __restrict__ bid, const int32_t* __restrict__ topk, int k,
                       int64_t n_q, KvMap kv, float scale_log2, float* __restrict__ lse,
                       const int32_t* __restrict__ order) {
  using namespace pair;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const uint32_t warp = warp_id(), lane = lane_id();
  const uint32_t crank = cluster_ctarank();
  const uint32_t peer = crank ^ 1u;
  const int64_t cluster = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;
  const int n_my = static_cast<int>((n_q - cluster + n_clusters - 1) / n_clusters);  // queries
  // Query of this pair's n-th slot: slot cluster + n * n_clusters of the schedule (`order`, a
  // permutation of the queries; the identity when null).
  auto query = [&](int n) {
    const int64_t i = cluster + static_cast<int64_t>(n) * n_clusters;
    return order != nullptr ? static_cast<int64_t>(__ldg(order + i)) : i;
  };
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + kOffAbort);
  volatile int* nt_buf = reinterpret_cast<volatile int*>(smem + kOffNT);
  auto bar = [&](int i) { return sbase + kOffBar + 8u * static_cast<uint32_t>(i); };
  // CTA 1 has no S tiles, Q or courier: it reuses the first S barrier as its o_drained.
  const int kOD = kSFull;

  const bool aligned = (sbase & 1023u) == 0;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(kKvFull + i), 32 * kGatherPerSlot);   // every gather warp of the slot
      mbar_init(bar(kKvEmpty + i), 1);
    }
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(kSFull + i), (crank == 0 || i > 0) ? 1 : 4);  // CTA 1: first = o_drained
      mbar_init(bar(kSEmpty + i), 4);
    }
    for (int i = 0; i < kPBuf; ++i) {
      mbar_init(bar(kPStaged + i), 128);
      mbar_init(bar(kPSEmpty + i), 1);
      mbar_init(bar(kPFull + i), 1);
      mbar_init(bar(kPEmpty + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kMetaFull + i), 1);
      mbar_init(bar(kMetaEmpty + i),
                crank == 0 ? kGatherPerSlot * kStages + 6 : kGatherPerSlot * kStages + 5);
      mbar_init(bar(kLReady + i), 1);               // CTA 1: armed with 512 tx bytes per query
      mbar_init(bar(kLEmpty + i), 128);
    }
    mbar_init(bar(kQFree), 1);                      // CTA 0: every QK of a query complete
    mbar_init(bar(kCorrGo), 1);
    mbar_init(bar(kCorrReady), 1);
    mbar_init(bar(kCorrDone), 128);
    mbar_init(bar(kOFinal), 1);
    *abort_flag = aligned ? 0u : 1u;
    if (!aligned) report_device_error(kErrBadIndex | 0xB2u);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc<512>(sbase + kOffTmem);
  __syncthreads();
  cluster_sync();                                    // the peer's barriers exist from here on
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffTmem);

  // meta_empty arrivals per query: CTA 0: every gather warp + QK + courier + 4 softmax warps
  // (at the end of the query: they read the masks until then); CTA 1: every gather warp + PV +
  // 4 row warps.
  auto meta_wait = [&](int n, bool warp_uniform) -> int {
    const uint32_t mb = bar(kMetaFull + (n & 1)), par = (n >> 1) & 1;
    const bool ok = warp_uniform ? warp_wait(mb, par, 0x40, abort_flag)
                                 : mbar_wait(mb, par, 0x40, abort_flag);
    return ok ? nt_buf[n & 1] : -1;
  };

  if (warp == kMetaWarp) {
    if (lane == 0 && crank == 0) tma_prefetch_desc(&tm_q);
    // ---------------------------------------------------------------- query metadata
    // Tile count (tiles up to the last valid entry) and, in CTA 0, the per-tile validity masks
    // of each query, two queries ahead; also pulls the query's Q rows into L2.
    for (int n = 0; n < n_my; ++n) {
      if (!warp_wait(bar(kMetaEmpty + (n & 1)), ((n >> 1) & 1) ^ 1, 0x41, abort_flag)) break;
      const int64_t t = query(n);
      const int32_t* trow = topk + t * k;
      const int bq = __ldg(bid + t);
      const int lim = (bq >= 0 && bq < kv.n_req) ? entry_limit(kv, bq, t) : -1;
      bool bad_entry = false;
      if (crank == 0) {
        const char* qrow = reinterpret_cast<const char*>(q + t * kH * kDQK);
        for (int off = static_cast<int>(lane) * 128; off < kH * kDQK * 2; off += 32 * 128)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(qrow + off));
      }
      uint32_t* mwords = reinterpret_cast<uint32_t*>(smem + kOffMask) + (n & 1) * kMaskWords;
      const int n_tiles_max = (k + kKeys - 1) / kKeys;
      int last = 0;
      for (int base = 0; base < n_tiles_max * kKeys; base += 32 * 8) {
        const int e0 = base + static_cast<int>(lane) * 8;
        uint32_t bits = 0;
        if (e0 + 8 <= k && (k & 3) == 0) {
          const int4 a = __ldg(reinterpret_cast<const int4*>(trow + e0));
          const int4 b4 = __ldg(reinterpret_cast<const int4*>(trow + e0 + 4));
          const int v[8] = {a.x, a.y, a.z, a.w, b4.x, b4.y, b4.z, b4.w};
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            bits |= (v[i] >= 0 && v[i] <= lim ? 1u : 0u) << i;
            bad_entry |= v[i] > lim;
          }
        } else {
          for (int i = 0; i < 8; ++i) {
            const int v = e0 + i < k ? __ldg(trow + e0 + i) : -1;
            bits |= (v >= 0 && v <= lim ? 1u : 0u) << i;
            bad_entry |= v > lim;
          }
        }
        const uint32_t w = bits << ((lane & 3) * 8);           // 4 lanes -> one 32-bit word
        const uint32_t w2 = w | __shfl_xor_sync(0xffffffffu, w, 1);
        const uint32_t word = w2 | __shfl_xor_sync(0xffffffffu, w2, 2);
        if ((lane & 3) == 0 && e0 < n_tiles_max * kKeys) {
          if (crank == 0) mwords[e0 / 32] = word;
          if (word) last = (e0 + 31 - __clz(word)) / kKeys + 1;
        }
      }
      last = __reduce_max_sync(0xffffffffu, last);
      if (__any_sync(0xffffffffu, bad_entry) && lane == 0 && crank == 0)
        report_device_error(kErrBadIndex);
      if (lane == 0) {
        nt_buf[n & 1] = last;
        mbar_arrive(bar(kMetaFull + (n & 1)));
      }
      __syncwarp();
    }
  } else if ((warp >= kGatherWarp0 && warp < kGatherWarp0 + kStages) ||
             (warp >= kGatherWarp1 && warp < kGatherWarp1 + (kGatherPerSlot - 1) * kStages)) {
    // ---------------------------------------------------------------- row gather (both CTAs)
    // kGatherPerSlot warps fill ring slot s with the global tiles g = s (mod kStages), an equal
    // share of the rows each: 16-byte cp.async copies into the 128B-swizzled K-major layout (row
    // r of atom a at a * kAtomBytes + r * 128, 16-byte chunk c at (c ^ (r % 8)) * 16); each
    // waits for its own copies, fences them for the tensor core (async proxy) and arrives.
    const int gi = warp >= kGatherWarp1 ? static_cast<int>(warp) - kGatherWarp1 + kStages
                                        : static_cast<int>(warp) - kGatherWarp0;
    const int half = gi / kStages;                   // this warp's share of the slot's rows
    const int s = gi % kStages;
    const int n_atoms = crank == 0 ? kAtomsS : kAtomsO;
    const uint32_t stage = sbase + s * (crank == 0 ? kStageS : kStageO);
    const int chunk = static_cast<int>(lane & 7);
    bool bad = false;
    int64_t q_tma_rp = -1;                           // ring position of this lane's last Q load
    // Ring entries of a query: CTA 0 first its kQPieces Q pieces (not for a query without
    // keys), then its key tiles; CTA 1 only the tiles (V). rpos0 = ring position of the query's
    // first entry; slot s takes the positions = s (mod kStages).
    int64_t rpos0 = 0;
    for (int n = 0; n < n_my && !*abort_flag; ++n) {
      const int nt = meta_wait(n, true);
      if (nt < 0) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kMetaEmpty + (n & 1)));
      const int64_t t = query(n);
      const int32_t* trow = topk + t * k;
      const int b = __ldg(bid + t);
      const bool b_ok = b >= 0 && b < kv.n_req;
      bad |= !b_ok;
      const int bb = b_ok ? b : 0;
      const int lim = b_ok ? entry_limit(kv, b, t) : -1;
      const int n_pre = (crank == 0 && nt > 0) ? kQPieces : 0;
      const int n_ent = n_pre + nt;
      const int e_first = static_cast<int>(((s - rpos0) % kStages + kStages) % kStages);
      auto fetch = [&](int j, int& s0, int& s1) {
        const int e0 = j * kKeys + static_cast<int>(lane);
        s0 = (j >= 0 && j < nt && e0 < k && b_ok) ? __ldg(trow + e0) : -1;
        s1 = (j >= 0 && j < nt && lane < kKeys - 32 && e0 + 32 < k && b_ok) ? __ldg(trow + e0 + 32) : -1;
      };
      int s0, s1;
      {                                              // first key tile this warp gathers
        int e = e_first;
        while (e < n_pre) e += kStages;
        fetch(e - n_pre, s0, s1);
      }
      bool ok = true;
      for (int e = e_first; e < n_ent; e += kStages) {
        const int64_t rp = rpos0 + e;
        if (!warp_wait(bar(kKvEmpty + s), static_cast<uint32_t>(((rp / kStages) & 1) ^ 1), 0x21,
                       abort_flag)) { ok = false; break; }
        if (e < n_pre) {
          // Q piece e: rows 0..127 (heads) of q[t], atoms kQAtomsPerPiece*e .. +2, each one TMA
          // box of 128 rows x 64 dims in the 128B-swizzled layout; the bytes complete on the
          // slot's full barrier next to the warps' usual arrivals (the byte count is added
          // without an arrival of its own, before this lane's arrival below)
          if (half == 0 && lane == 0) {
            mbar_add_tx(bar(kKvFull + s), kQAtomsPerPiece * kQAtomBytes);
#pragma unroll
            for (int a = 0; a < kQAtomsPerPiece; ++a)
              tma_load_2d(stage + a * kQAtomBytes, &tm_q, (e * kQAtomsPerPiece + a) * 64,
                          static_cast<int32_t>(t * kH), bar(kKvFull + s));
            q_tma_rp = rp;
          }
        } else {
          const int j = e - n_pre;
          const int32_t r0 = kv_row(kv, bb, s0, lim, &bad);
          const int32_t r1 = kv_row(kv, bb, s1, lim, &bad);
          fetch(j + kStages, s0, s1);
#pragma unroll
          for (int i = half; i < kKeys / 4; i += kGatherPerSlot) {
            const int r = static_cast<int>(lane >> 3) + 4 * i;        // tile row of this lane
            const int32_t ra = __shfl_sync(0xffffffffu, r0, r & 31);
            const int32_t rb = __shfl_sync(0xffffffffu, r1, r & 31);
            const int32_t row = r < 32 ? ra : rb;
            const bool valid = row < kv.n_rows;
            const __nv_bfloat16* src = c + (valid ? static_cast<int64_t>(row) * kDQK : 0) + chunk * 8;
            const uint32_t dst = stage + r * 128 + ((chunk ^ (r & 7)) * 16);   // r & 7: atoms are 1 KB aligned
            for (int a = 0; a < n_atoms; ++a)
              cp_async16(dst + a * kAtomBytes, src + a * 64, valid ? 16u : 0u);
          }
        }
        cp_async_commit();
        cp_async_wait_all();
        fence_proxy_async_smem();
        mbar_arrive(bar(kKvFull + s));
      }
      if (!ok) break;
      rpos0 += n_ent;
    }
    cp_async_wait_all();
    if (*abort_flag && q_tma_rp >= 0) {
      // unwinding: let this lane's last Q load land before the CTA can exit (bounded)
      const long long t0 = clock64();
      while (!mbar_try_wait(bar(kKvFull + s), static_cast<uint32_t>((q_tma_rp / kStages) & 1)) &&
             clock64() - t0 < kWaitLimitCycles) {
      }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) report_device_error(kErrBadIndex);
  } else if (warp == kMmaWarp && crank == 0) {
    // ---------------------------------------------------------------- CTA 0: QK issuer
    // Tile g: ring slot g % kStages -> S buffer g % kStages. The whole warp runs the loop
    // (waits and descriptor arithmetic stay warp-uniform) and one elected lane issues: an MMA
    // issued this way leaves the issuing thread at the tensor pipe's own rate, about twice as
    // fast as from a single-lane branch.
    const bool leader = elect_one();
    const uint32_t idesc = idesc_bf16(128, kKeys, 0, 0);
    const uint64_t desc0 = smem_desc(sbase, 16, 1024, kSwizzle128B);
    int rs = 0, sb = 0;                              // ring slot of the next entry; S buffer
    uint32_t r_ph = 0, s_ph = 0;                     // ... and the parity of their current use
    bool ok = true;
    for (int n = 0; n < n_my && ok; ++n) {
      const int nt = meta_wait(n, true);
      if (nt < 0) break;
      __syncwarp();
      if (leader) mbar_arrive(bar(kMetaEmpty + (n & 1)));
      const int n_pre = nt > 0 ? kQPieces : 0;
      // Q pieces -> TMEM columns kColQ.. (the A operand of QK), once every QK MMA and copy of
      // the previous query is complete (kQFree; an MMA issued after a copy by this thread sees it).
      for (int pce = 0; pce < n_pre; ++pce) {
        const int s = rs;
        if (!warp_wait(bar(kKvFull + s), r_ph, 0x22, abort_flag)) { ok = false; break; }
        if (pce == 0 && n > 0 &&
            !warp_wait(bar(kQFree), static_cast<uint32_t>((n - 1) & 1), 0x25, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (leader) {
          const uint64_t dq = desc0 + static_cast<uint64_t>((s * kStageS) >> 4);
#pragma unroll
          for (int a = 0; a < kQAtomsPerPiece; ++a)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)           // 16 dims (8 columns) per copy
              tmem_cp_128x256b(tmem + kColQ + (pce * kQAtomsPerPiece + a) * 32 + kk * 8,
                               dq + static_cast<uint64_t>((a * kQAtomBytes + kk * 32) >> 4));
          umma_commit(bar(kKvEmpty + s));            // the slot is free once the copies read it
        }
        __syncwarp();
        if (++rs == kStages) { rs = 0; r_ph ^= 1u; }
      }
      if (!ok) break;
      tc_fence_after();
      for (int j = 0; j < nt; ++j) {
        const int s = rs;
        const uint32_t d_s = tmem + kColS + sb * kSStride;
        if (!warp_wait(bar(kKvFull + s), r_ph, 0x23, abort_flag)) { ok = false; break; }
        if (!warp_wait(bar(kSEmpty + sb), s_ph ^ 1u, 0x24, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint64_t db0 = desc0 + static_cast<uint64_t>((s * kStageS) >> 4);
#pragma unroll
        for (int gg = 0; gg < kDQK / 16; ++gg) {
          const uint64_t db =
              db0 + static_cast<uint64_t>(((gg >> 2) * kAtomBytes + (gg & 3) * 32) >> 4);
          if (leader) umma_ts(d_s, tmem + kColQ + gg * 8, db, idesc, gg > 0 ? 1u : 0u);
        }
        if (leader) {
          umma_commit(bar(kSFull + sb));
          umma_commit(bar(kKvEmpty + s));          // the slot is free once these MMAs finish
        }
        __syncwarp();
        if (++rs == kStages) { rs = 0; r_ph ^= 1u; }
        if (++sb == kStages) { sb = 0; s_ph ^= 1u; }
      }
      if (leader) umma_commit(bar(kQFree));        // Q of this query no longer read
      __syncwarp();
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      // -------------------------------------------------------------- CTA 1: PV issuer
      const uint32_t idesc = idesc_bf16(128, 256, 0, 1);
      volatile int* corr_j = reinterpret_cast<volatile int*>(smem + kOffCorrJ);
      const uint64_t p_desc0 = smem_desc(sbase + kOffP, 16, 256, kSwizzle32B);
      const uint64_t v_desc0 = smem_desc(sbase, kAtomBytes, 1024, kSwizzle128B);
      uint32_t n_ev = 0;
      bool ok = true;
      // each P buffer always has one armed delivery (one bulk copy of P + alpha + flags)
      for (int i = 0; i < kPBuf; ++i) mbar_expect_tx(bar(kPFull + i), kPBytes + kAFBytes);
      int s = 0, pb = 0;                             // ring slot and P buffer of the tile
      uint32_t r_ph = 0, p_ph = 0;                   // ... and the parity of their current use
      for (int n = 0; n < n_my && ok; ++n) {
        const int nt = meta_wait(n, false);
        if (nt < 0) break;
        mbar_arrive(bar(kMetaEmpty + (n & 1)));
        // O of the previous query must be drained before this query overwrites it
        if (n > 0 && !mbar_wait(bar(kOD), (n - 1) & 1, 0x32, abort_flag)) break;
        tc_fence_after();
        for (int j = 0; j < nt && ok; ++j) {
          if (!mbar_wait(bar(kKvFull + s), r_ph, 0x25, abort_flag)) { ok = false; break; }
          if (!mbar_wait(bar(kPFull + pb), p_ph, 0x26, abort_flag)) { ok = false; break; }
          mbar_expect_tx(bar(kPFull + pb), kPBytes + kAFBytes);
          const volatile uint32_t* flags =
              reinterpret_cast<const volatile uint32_t*>(smem + kOffAlpha + pb * kAFStride + 512);
          if (flags[0] | flags[1] | flags[2] | flags[3]) {
            // a row's reference maximum moved: the row warps rescale O after the previous PV
            *corr_j = static_cast<int>(pb);
            umma_commit(bar(kCorrReady));
            mbar_arrive(bar(kCorrGo));
            if (!mbar_wait(bar(kCorrDone), n_ev & 1u, 0x27, abort_flag)) { ok = false; break; }
            ++n_ev;
          }
          tc_fence_after();
          const uint64_t da0 = p_desc0 + static_cast<uint64_t>((pb * kPBytes) >> 4);
          const uint64_t dv0 = v_desc0 + static_cast<uint64_t>((s * kStageO) >> 4);
#pragma unroll
          for (int kk = 0; kk < kKeys / 16; ++kk) {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
              umma_ss(tmem + hf * 256, da0 + static_cast<uint64_t>((kk * kPAtomBytes) >> 4),
                      dv0 + static_cast<uint64_t>((hf * 4 * kAtomBytes + kk * 2048) >> 4), idesc,
                      (j > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit_multicast(bar(kPEmpty + pb), static_cast<uint16_t>(1u << peer));
          umma_commit(bar(kKvEmpty + s));
          if (++s == kStages) { s = 0; r_ph ^= 1u; }
          if (++pb == kPBuf) { pb = 0; p_ph ^= 1u; }
        }
        if (!ok) break;
        umma_commit(bar(kOFinal));                   // O of this query complete
        *corr_j = -1;                                // end of this query's rescale requests
        mbar_arrive(bar(kCorrGo));
      }
    }
  } else if (warp == kCourierWarp) {
    if (lane == 0 && crank == 0) {
      // -------------------------------------------------------------- CTA 0: P courier
      // Ships each staged P tile (+ alpha, flags) to CTA 1 with two bulk copies that complete
      // on CTA 1's p_full barrier, then hands the staging buffer back to the softmax warps.
      int pb = 0;                                    // P buffer of the tile
      uint32_t pph = 0;                              // ... and the parity of its current use
      for (int n = 0; n < n_my; ++n) {
        const int nt = meta_wait(n, false);
        if (nt < 0) break;
        mbar_arrive(bar(kMetaEmpty + (n & 1)));
        bool ok = true;
        for (int j = 0; j < nt; ++j) {
          if (!mbar_wait(bar(kPStaged + pb), pph, 0x2E, abort_flag)) { ok = false; break; }
          if (!mbar_wait(bar(kPEmpty + pb), pph ^ 1u, 0x2F, abort_flag)) { ok = false; break; }
          const uint32_t src = sbase + kOffPS + pb * kPSStride;
          bulk_copy_to_peer(sbase + kOffP + pb * kPBytes, src, kPBytes, bar(kPFull + pb), peer);
          bulk_copy_to_peer(sbase + kOffAlpha + pb * kAFStride, src + kPBytes, kAFBytes,
                            bar(kPFull + pb), peer);
          bulk_commit();
          bulk_wait_read_all();
          mbar_arrive(bar(kPSEmpty + pb));
          if (++pb == kPBuf) { pb = 0; pph ^= 1u; }
        }
        if (!ok) break;
      }
      bulk_wait_all();                               // every copy to the peer has landed
    }
  } else if (crank == 0 && warp < 4) {
    // ---------------------------------------------------------------- CTA 0: softmax warps
    const int h = static_cast<int>(threadIdx.x);
    const uint32_t lane_base = (warp * 32u) << 16;
    int sb = 0, psb = 0;                             // S buffer and P staging buffer of the tile
    uint32_t s_ph = 0, ps_ph = 0;                    // ... and the parity of their current use
    for (int n = 0; n < n_my; ++n) {
      const int nt = meta_wait(n, true);
      if (nt < 0) break;
      const int64_t t = query(n);
      const uint32_t* mwords = reinterpret_cast<const uint32_t*>(smem + kOffMask) + (n & 1) * kMaskWords;
      float m_ref = -INFINITY, l_run = 0.f;
      bool ok = true;
      for (int j = 0; j < nt; ++j) {
        if (!warp_wait(bar(kSFull + sb), s_ph, 0x28, abort_flag)) { ok = false; break; }
        tc_fence_after();
        float sv[kKeys];
        {
          uint32_t r[32], r16[16];                   // both loads in flight, one wait
          tmem_ld32(tmem + lane_base + kColS + sb * kSStride, r);
          tmem_ld16(tmem + lane_base + kColS + sb * kSStride + 32, r16);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) sv[i] = __uint_as_float(r[i]);
#pragma unroll
          for (int i = 0; i < kKeys - 32; ++i) sv[32 + i] = __uint_as_float(r16[i]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kSEmpty + sb));
        const int e0 = j * kKeys;                    // validity bits of this tile's entries
        const uint64_t mk = ((static_cast<uint64_t>(mwords[(e0 >> 5) + 1]) << 32) |
                             mwords[e0 >> 5]) >> (e0 & 31);
        const uint32_t mlo = static_cast<uint32_t>(mk), mhi = static_cast<uint32_t>(mk >> 32);
        const bool full = mlo == 0xFFFFFFFFu && (mhi & 0xFFFFu) == 0xFFFFu;   // common case
        auto valid_at = [&](int i) {
          return full || (i < 32 ? ((mlo >> i) & 1u) != 0u : ((mhi >> (i - 32)) & 1u) != 0u);
        };
        // x_i = scale * s_i - m_ref in the log2 domain (one FMA); masked entries -inf, whose
        // ex2 is 0. m_ref moves only when a row's maximum x grows above kLazyLog2. The common
        // case takes no maximum: p = 2^x against the current m_ref, and since the row's sum of p
        // bounds its largest p, only a sum of at least 2^(kLazyLog2 - 1) (an x above
        // kLazyLog2 - 1) looks at the maximum and, if it moved, redoes p.
        float alpha = 1.f;
        if (m_ref == -INFINITY) {                    // no valid entry in this row so far
          float mt = -INFINITY;
#pragma unroll
          for (int i = 0; i < kKeys; ++i) {
            sv[i] = valid_at(i) ? sv[i] * scale_log2 : -INFINITY;
            mt = fmaxf(mt, sv[i]);
          }
          m_ref = mt;
          if (mt != -INFINITY) {
#pragma unroll
            for (int i = 0; i < kKeys; ++i) sv[i] -= mt;
          }
        } else if (full) {
          // every entry valid (the common case, the same for the whole warp): two-wide FMAs
          // without a per-entry mask test
          const float nm = -m_ref;
          const float2 sc2 = make_float2(scale_log2, scale_log2), nm2 = make_float2(nm, nm);
#pragma unroll
          for (int i = 0; i < kKeys; i += 2) {
            const float2 a = __ffma2_rn(make_float2(sv[i], sv[i + 1]), sc2, nm2);
            sv[i] = a.x; sv[i + 1] = a.y;
          }
        } else {
          const float nm = -m_ref;
#pragma unroll
          for (int i = 0; i < kKeys; ++i) sv[i] = valid_at(i) ? fmaf(sv[i], scale_log2, nm) : -INFINITY;
        }
        uint32_t pk[kKeys / 2];
        auto exp_pack = [&]() {                      // p = 2^x as bf16 pairs; returns sum p
          float sa = 0.f, sc = 0.f;
#pragma unroll
          for (int i = 0; i < kKeys; i += 2) {
            const float p0 = ex2_approx(sv[i]), p1 = ex2_approx(sv[i + 1]);
            sa += p0;
            sc += p1;
            pk[i / 2] = bf16x2_bits(p0, p1);
          }
          return sa + sc;
        };
        float psum = exp_pack();
        if (!(psum < kLazySum)) {                    // rare (also taken by a NaN sum)
          float xm = -INFINITY;
#pragma unroll
          for (int i = 0; i < kKeys; ++i) xm = fmaxf(xm, sv[i]);
          if (xm > kLazyLog2) {                      // move the reference maximum
            alpha = ex2_approx(-xm);
            m_ref += xm;
#pragma unroll
            for (int i = 0; i < kKeys; ++i) sv[i] -= xm;
            psum = exp_pack();
          }
        }
        l_run = l_run * alpha + psum;
        const uint32_t any = __any_sync(0xffffffffu, alpha != 1.f) ? 1u : 0u;
        // Stage P (swizzled K-major rows), alpha and the warp flags in staging buffer psb
        // once the courier has shipped its previous contents.
        if (!warp_wait(bar(kPSEmpty + psb), ps_ph ^ 1u, 0x29, abort_flag)) { ok = false; break; }
        uint8_t* slot = smem + kOffPS + psb * kPSStride;
        uint8_t* prow = slot + (h >> 3) * 256 + (h & 7) * 32;
        const int swz = (h >> 2) & 1;
#pragma unroll
        for (int cc = 0; cc < kKeys / 8; ++cc)       // chunk cc: keys 8cc..8cc+7, atom cc / 2
          *reinterpret_cast<uint4*>(prow + (cc >> 1) * kPAtomBytes + (((cc & 1) ^ swz) * 16)) =
              make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
        reinterpret_cast<float*>(slot + kPBytes)[h] = alpha;
        if (lane == 0) reinterpret_cast<uint32_t*>(slot + kPBytes + 512)[warp] = any;
        fence_proxy_async_smem();
        mbar_arrive(bar(kPStaged + psb));
        if (++sb == kStages) { sb = 0; s_ph ^= 1u; }
        if (++psb == kPBuf) { psb = 0; ps_ph ^= 1u; }
      }
      if (!ok) break;
      // l of this query -> CTA 1 (buffer n % 2, free once CTA 1 read query n - 2's) as an
      // asynchronous store that completes on CTA 1's l_ready barrier (no release fence, which
      // would first wait for every earlier memory operation of the thread), then lse
      if (n >= 2 && !warp_wait(bar(kLEmpty + (n & 1)), ((n >> 1) & 1) ^ 1, 0x43, abort_flag)) break;
      st_async_u32(sbase + kOffL + ((n & 1) * 128 + h) * 4, bar(kLReady + (n & 1)), peer,
                   __float_as_uint(l_run));
      if (lse != nullptr)
        lse[t * kH + h] = l_run > 0.f ? (m_ref + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kMetaEmpty + (n & 1)));
    }
  } else if (crank == 1 && warp < 4) {
    // ---------------------------------------------------------------- CTA 1: O rows
    const int h = static_cast<int>(threadIdx.x);
    const uint32_t lane_base = (warp * 32u) << 16;
    const volatile int* corr_j = reinterpret_cast<const volatile int*>(smem + kOffCorrJ);
    uint32_t n_go = 0, n_ev = 0;                     // corr_go completions, rescale events
    for (int n = 0; n < n_my; ++n) {
      const int nt = meta_wait(n, true);
      if (nt < 0) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kMetaEmpty + (n & 1)));
      const int64_t t = query(n);
      if (threadIdx.x == 0) mbar_expect_tx(bar(kLReady + (n & 1)), 128 * 4);   // l of query n
      bool ok = true;
      for (;;) {                                     // rescale requests, then the end marker
        if (!warp_wait(bar(kCorrGo), n_go & 1u, 0x2A, abort_flag)) { ok = false; break; }
        ++n_go;
        const int pb = *corr_j;
        if (pb < 0) break;
        if (!warp_wait(bar(kCorrReady), n_ev & 1u, 0x2B, abort_flag)) { ok = false; break; }
        ++n_ev;
        tc_fence_after();
        const float a = reinterpret_cast<const float*>(smem + kOffAlpha + pb * kAFStride)[h];
        if (__any_sync(0xffffffffu, a != 1.f)) {
#pragma unroll 1
          for (int c0 = 0; c0 < kDV; c0 += 16) {
            uint32_t r[16];
            tmem_ld16(tmem + lane_base + c0, r);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * a);
            tmem_st16(tmem + lane_base + c0, r);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(bar(kCorrDone));
      }
      if (ok) ok = warp_wait_cluster(bar(kLReady + (n & 1)), (n >> 1) & 1, 0x2C, abort_flag);
      if (ok) ok = warp_wait(bar(kOFinal), n & 1, 0x2D, abort_flag);
      if (!ok) break;
      tc_fence_after();
      const float l = reinterpret_cast<const volatile float*>(smem + kOffL)[(n & 1) * 128 + h];
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      // o = O / l in bf16, 64 columns per round: TMEM -> registers -> the warp's swizzled
      // staging tile -> one TMA store of 32 rows x 128 B (coalesced, asynchronous).
      // Two staging tiles per warp, alternating, so a store can still be reading one tile
      // while the next round fills the other.
      const uint32_t xo[2] = {static_cast<uint32_t>(kOffX + warp * (32 * 128)),
                              static_cast<uint32_t>(kOffXO1 + warp * (32 * 128))};
#pragma unroll 1
      for (int c0 = 0; c0 < kDV; c0 += 64) {
        const uint32_t xoff = xo[(c0 >> 6) & 1];
        uint8_t* xrow = smem + xoff + lane * 128;
        uint32_t r[64];
        if (nt > 0) {
          uint32_t (&ra)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[0]);
          uint32_t (&rb)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[32]);
          tmem_ld32(tmem + lane_base + c0, ra);
          tmem_ld32(tmem + lane_base + c0 + 32, rb);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 64; ++i) r[i] = 0u;
        }
        if (c0 + 64 == kDV) {                        // all of O read: PV may overwrite it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kOD));
        }
        if (lane == 0) bulk_wait_read_but_one();     // the store of two rounds ago read this tile
        __syncwarp();
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          uint32_t pk[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            pk[i] = bf16x2_bits(__uint_as_float(r[8 * v + 2 * i]) * inv_l,
                                __uint_as_float(r[8 * v + 2 * i + 1]) * inv_l);
          *reinterpret_cast<uint4*>(xrow + ((v ^ (lane & 7)) * 16)) =
              make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        fence_proxy_async_smem();                    // the tile is read by the TMA unit
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tm_o, sbase + xoff, c0, static_cast<int32_t>(t * kH + warp * 32));
          bulk_commit();
        }
      }
      // the l buffer may be refilled (query n + 2): every row read it; off the critical path
      mbar_arrive_cluster(bar(kLEmpty + (n & 1)), peer);
    }
    if (lane == 0) bulk_wait_all();                  // stores complete before the CTA exits
  }

  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc<512>(tmem);
  }
  cluster_sync();                                    // no CTA leaves while its peer may write
}

// Schedule for the persistent pairs: queries sorted by their number of key tiles, largest
// first (counting sort; a query at position p selects min(p + 1, k) keys), and dealt to the
// pairs in rounds whose direction alternates, so that the pairs' total work evens out. Slot i of
// the schedule is processed by pair i % n_pairs.
constexpr int kOrderThreads = 1024;
constexpr int kOrderBuckets = (kMaxK + pair::kKeys - 1) / pair::kKeys + 1;
__global__ void __launch_bounds__(kOrderThreads)
mla_order_kernel(const int32_t* __restrict__ pos, int k, int n_q, int n_pairs,
                 int32_t* __restrict__ order) {
  __shared__ uint32_t hist[kOrderBuckets], next[kOrderBuckets];
  for (int b = threadIdx.x; b < kOrderBuckets; b += blockDim.x) hist[b] = 0;
  __syncthreads();
  auto tiles_of = [&](int t) {
    const int p = __ldg(pos + t);
    const int sel = p < 0 ? 0 : (p >= k ? k : p + 1);
    return (sel + pair::kKeys - 1) / pair::kKeys;
  };
  for (int t = threadIdx.x; t < n_q; t += blockDim.x) atomicAdd(&hist[tiles_of(t)], 1u);
  __syncthreads();
  if (threadIdx.x == 0) {                            // bucket b starts after every larger bucket
    uint32_t run = 0;
    for (int b = kOrderBuckets - 1; b >= 0; --b) {
      next[b] = run;
      run += hist[b];
    }
  }
  __syncthreads();
  for (int t = threadIdx.x; t < n_q; t += blockDim.x) {
    const int p = static_cast<int>(atomicAdd(&next[tiles_of(t)], 1u));   // rank, largest first
    const int r = p / n_pairs;
    int j = p - r * n_pairs;
    if ((r & 1) && (r + 1) * n_pairs <= n_q) j = n_pairs - 1 - j;          // full rounds snake
    order[r * n_pairs + j] = t;
  }
}

int launch_mla_pair(const void* q, const void* c, int64_t n_kv_rows, const KvMap& kv,
                    const int32_t* bid, const int32_t* topk, int64_t n_q, int k, float scale,
                    void* o, float* lse, const int32_t* pos, int32_t* order_ws,
                    cudaStream_t stream) {
  (void)n_kv_rows;
  CUtensorMap tm_o, tm_q;                            // o as [n_q * 128 rows, 512 columns]
  int rc = make_tmap_bf16_2d(&tm_o, o, static_cast<uint64_t>(n_q) * pair::kH, pair::kDV,
                             pair::kDV * 2, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  rc = make_tmap_bf16_2d(&tm_q, q, static_cast<uint64_t>(n_q) * pair::kH, pair::kDQK,
                         pair::kDQK * 2, 64, pair::kH, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;                                 // q as [n_q * 128 rows, 576 columns]
  DSA_CHECK_CUDA(cudaFuncSetAttribute(sparse_mla_pair_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, pair::kSmem));
  const int64_t pairs = std::min<int64_t>(n_q, num_sms_cached() / 2);
  const int32_t* order = nullptr;
  if (pos != nullptr && order_ws != nullptr) {
    mla_order_kernel<<<1, kOrderThreads, 0, stream>>>(pos, k, static_cast<int>(n_q),
                                                      static_cast<int>(pairs), order_ws);
    DSA_CHECK_CUDA(cudaGetLastError());
    order = order_ws;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(pairs * 2));
  cfg.blockDim = dim3(pair::kThreads);
  cfg.dynamicSmemBytes = pair::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const float scale_log2 = scale * 1.4426950408889634f;
  DSA_CHECK_CUDA(cudaLaunchKernelEx(&cfg, sparse_mla_pair_kernel, tm_o, tm_q,
                                    static_cast<const __nv_bfloat16*>(c),
                                    static_cast<const __nv_bfloat16*>(q), bid, topk, k, n_q, kv,
                                    scale_log2, lse, order));
  return DSA_OK;
}

template <int H, int DQK, int DV>
int launch_mla(const void* q, const void* c, int64_t n_kv_rows, const KvMap& kv,
               const int32_t* bid, const int32_t* topk, int64_t n_q, int k, float scale,
               void* o, float* lse, cudaStream_t stream) {
  using S = MlaShape<H, DQK, DV>;
  CUtensorMap tc;
  int rc = make_tmap_bf16_2d(&tc, c, static_cast<uint64_t>(n_kv_rows), DQK, DQK * 2, 64, 1,
                             CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  auto kern = sparse_mla_kernel<H, DQK, DV>;
  DSA_CHECK_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmem));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(n_q));
  cfg.blockDim = dim3(S::kThreads);
  cfg.dynamicSmemBytes = S::kSmem;
  cfg.stream = stream;
  const float scale_log2 = scale * 1.4426950408889634f;
  DSA_CHECK_CUDA(cudaLaunchKernelEx(&cfg, kern, tc, static_cast<const __nv_bfloat16*>(q), bid, topk,
                                    k, kv, scale_log2, static_cast<__nv_bfloat16*>(o), lse));
  return DSA_OK;
}

}  // namespace

size_t sparse_mla_workspace_bytes(int64_t n_q) {
  return n_q > 0 ? static_cast<size_t>(n_q) * sizeof(int32_t) : 0;
}

int sparse_mla(const void* q, const void* c, int64_t n_kv_rows, const int32_t* cu, int n_req,
               const int32_t* bid, const int32_t* topk, int64_t n_q, int H, int dqk, int dv, int k,
               float scale, const int32_t* block_table, int max_pages, int page_size, void* o,
               float* lse, const int32_t* pos, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (n_q < 0 || k < 1 || n_kv_rows < 0 || n_req < 1)
    return fail(DSA_ERR_INVALID, "mla: need n_q >= 0, k >= 1, n_kv_rows >= 0, n_req >= 1");
  if (n_q == 0) return DSA_OK;
  if (!q || !c || !bid || !topk || !o) return fail(DSA_ERR_INVALID, "mla: null pointer");
  if (!block_table && !cu) return fail(DSA_ERR_INVALID, "mla: need cu or block_table");
  if (block_table && (page_size != kPageRows || max_pages < 1))
    return fail(DSA_ERR_UNSUPPORTED, "mla: paged KV needs page_size 64 (got %d)", page_size);
  if (k > kMaxK) return fail(DSA_ERR_UNSUPPORTED, "mla: k = %d > %d", k, kMaxK);
  if (n_kv_rows >= (1ll << 31) || n_q * static_cast<int64_t>(H) >= (1ll << 31))
    return fail(DSA_ERR_UNSUPPORTED, "mla: sizes beyond 32-bit TMA coordinates");
  if (reinterpret_cast<uintptr_t>(q) % 16 || reinterpret_cast<uintptr_t>(o) % 16)
    return fail(DSA_ERR_INVALID, "mla: q and o must be 16-byte aligned");
  if (pos != nullptr && (ws == nullptr || ws_bytes < sparse_mla_workspace_bytes(n_q)))
    return fail(DSA_ERR_WORKSPACE, "mla: workspace of %zu bytes < %zu", ws_bytes,
                sparse_mla_workspace_bytes(n_q));
  if (ws != nullptr && reinterpret_cast<uintptr_t>(ws) % 16 != 0)
    return fail(DSA_ERR_INVALID, "mla: workspace must be 16-byte aligned");
  KvMap kv{cu, block_table, max_pages, n_req, n_kv_rows, pos};
  if (H == 128 && dqk == 576 && dv == 512)
    return launch_mla_pair(q, c, n_kv_rows, kv, bid, topk, n_q, k, scale, o, lse, pos,
                           static_cast<int32_t*>(ws), stream);
  if (H == 8 && dqk == 80 && dv == 64)
    return launch_mla<8, 80, 64>(q, c, n_kv_rows, kv, bid, topk, n_q, k, scale, o, lse, stream);
  return fail(DSA_ERR_UNSUPPORTED, "mla: (H, dqk, dv) = (%d, %d, %d) not built; supported "
                                   "(128, 576, 512), (8, 80, 64)", H, dqk, dv);
}

cudaError_t mla_read_errors(uint32_t* flags) { return read_and_clear_device_error(flags); }

}  // namespace dsa
