// Lightning-indexer scores on tcgen05 tensor cores.
//
//   I[t, s] = sum_h w[t, h] * ReLU( q_idx[t, h, :] . k_idx[row(b_t, s), :] ),  0 <= s <= pos_t
//
// "[RFC]: Parallel strategy for Deepseek v3.2 like models" (comments) names this history scan
// the model's bottleneck; sequence sharding divides it by sp. Design for sm_103a:
//
//  * The contraction is D[s, (t,h)] = K[s, :] . Q[(t,h), :] with the KEYS on the UMMA M side
//    (128 keys per tile, one TMEM lane each) and (query, head) pairs on N. Every epilogue
//    thread then owns one key and reduces its row over heads entirely in registers:
//    sum_h w[t,h] * max(D, 0). Per-head logits never leave TMEM; only the head-reduced fp32
//    score reaches global memory.
//  * One CTA works on a "group" of up to 2 x 256/Hi consecutive queries of one request
//    (8 queries for Hi = 64). Their Q rows (512 x Di bf16) stay in shared memory while the key
//    tiles stream through a 3-stage TMA ring. Each key tile feeds two MMAs (queries 0-3 and
//    4-7) into two TMEM accumulators of 256 fp32 columns, so one key tile is reused by 8
//    queries and the second accumulator's MMA hides the first one's epilogue.
//  * Warp roles: warps 0-3 and 4-7 are the epilogues of accumulators 0 and 1 (TMEM lane
//    quadrant = warp % 4), warp 8 issues TMA, warp 9 issues tcgen05.mma.
//  * Persistent grid (one CTA per SM). A one-CTA planning kernel cuts the queries into groups
//    (never across a request, at most 8 queries) and counts each group's causal 128-key tiles
//    (none when the caller only needs the scores of histories longer than some k, and no query
//    of the group has one: a top-k then takes every key of such a query whatever its scores);
//    the groups' tiles, concatenated in order, are split into equal contiguous ranges, one per
//    CTA (a range covers one or a few groups, so each CTA loads few Q blocks). Only tiles that
//    hold some causal key are computed; keys past a query's position are masked in the
//    epilogue.
//  * Key rows: contiguous (cu[b] + s, the logical order after the rerange) or paged
//    (block_table, 64-token pages, one TMA box per page).
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "keys.cuh"
#include "ptx.cuh"
#include "status.cuh"
#include "tmap.cuh"

namespace dsa {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kKeysPerTile = 128;
constexpr int kPageRows = 64;          // TMA box height for keys (also the page size)

struct Plan {
  int total_tiles;   // key tiles of all groups
  int pad;
  int n_groups;
  int error;
};

// Workspace carving for the schedule (scores, when owned by the workspace, follow it).
struct PlanLayout {
  size_t plan_off, groups_off, unit_off, t0_off, bytes;
  explicit PlanLayout(int64_t n_q) {
    auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    const size_t nq = static_cast<size_t>(n_q > 0 ? n_q : 1);
    plan_off = 0;
    groups_off = up(sizeof(Plan));
    unit_off = up(groups_off + nq * sizeof(int4));
    t0_off = up(unit_off + (nq + 1) * sizeof(int32_t));
    bytes = up(t0_off + nq * sizeof(int32_t));
  }
};

// F8: q_idx / k_idx rows are E4M3 codes (1 byte each) with fp32 scales, the MMA kind::f8f6f4
// (32 elements per instruction); otherwise bf16 rows and kind::f16 (16 per instruction). Either
// way one instruction consumes 32 bytes of each operand row.
template <int HI, int DI, bool F8 = false>
struct Shape {
  static constexpr int kEB = F8 ? 1 : 2;                 // bytes per element
  static constexpr int kQPA = 256 / HI;                  // queries per accumulator
  static constexpr int kGQ = 2 * kQPA;                   // queries per group
  static constexpr int kBRows = kGQ * HI;                // 512 rows of Q per group
  static constexpr int kRowBytes = DI * kEB;
  static constexpr int kAtomBytes = kRowBytes >= 128 ? 128 : kRowBytes;  // swizzled row bytes
  static constexpr int kAtomElems = kAtomBytes / kEB;
  static constexpr int kAtoms = DI / kAtomElems;
  static constexpr uint32_t kSwz = kAtomBytes == 128 ? kSwizzle128B : kSwizzle64B;
  static constexpr CUtensorMapSwizzle kTmaSwz =
      kAtomBytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  static constexpr CUtensorMapDataType kTmaType =
      F8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  static constexpr int kSBO = 8 * kAtomBytes;            // 8-row core-matrix group stride
  static constexpr int kAStage = kKeysPerTile * kRowBytes;
  static constexpr int kAAtom = kKeysPerTile * kAtomBytes;
  static constexpr int kBAtom = kBRows * kAtomBytes;
  static constexpr int kStages = F8 ? 4 : (DI >= 64 ? 3 : 4);
  static constexpr int kBBytes = kBRows * kRowBytes;
  static constexpr int kKSteps = kRowBytes / 32;
  static constexpr int kStepsPerAtom = kAtomBytes / 32;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kStages * kAStage;
  static constexpr int kOffW = kOffB + kBBytes;          // fp32 [kGQ][HI]
  static constexpr int kOffPos = kOffW + kGQ * HI * 4;   // int32 [kGQ]
  static constexpr int kOffBar = (kOffPos + kGQ * 4 + 7) & ~7;
  static constexpr int kNumBars = 2 * kStages + 10;
  static constexpr int kOffTmem = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffTmem + 4;
  static constexpr int kSmem = kOffAbort + 4;
  static constexpr int kThreads = 320;                   // 8 epilogue warps + TMA + MMA
  static_assert(kSmem <= 232448, "shared memory budget");
  static_assert(kOffB % 1024 == 0 && kAStage % 1024 == 0 && kBAtom % 1024 == 0, "alignment");
};

// ------------------------------------------------------------------------------------------
// Planning: groups of <= GQ consecutive queries of one request, and their key-tile counts.
__device__ __forceinline__ uint32_t plan_scan(uint32_t v, uint32_t* wt, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kW = kPlanThreads / 32;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wt[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < kW ? wt[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    wt[lane] = w;
  }
  __syncthreads();
  const uint32_t before = (warp > 0 ? wt[warp - 1] : 0u) + x - v;
  *total = wt[kW - 1];
  __syncthreads();
  return before;
}

__global__ void __launch_bounds__(kPlanThreads)
indexer_plan_kernel(const int32_t* __restrict__ pos, const int32_t* __restrict__ bid, int n_q,
                    int n_req, int max_ctx, int gq, int skip_le, Plan* plan, int4* groups,
                    int32_t* unit_start, int32_t* t0_list) {
  // key tiles of a group whose last position is pmax (none for an empty group, or when every
  // query's history pos + 1 is at most skip_le)
  auto group_tiles = [&](int pmax) {
    return pmax >= 0 && pmax + 1 > skip_le ? static_cast<uint32_t>(pmax / kKeysPerTile + 1) : 0u;
  };
  __shared__ uint32_t wt[32];
  const int per = (n_q + kPlanThreads - 1) / kPlanThreads;
  const int lo = min(static_cast<int>(threadIdx.x) * per, n_q), hi = min(lo + per, n_q);
  auto starts = [&](int t) {
    return t == 0 || (t % gq) == 0 || __ldg(bid + t) != __ldg(bid + t - 1);
  };
  uint32_t cnt = 0;
  for (int t = lo; t < hi; ++t) cnt += starts(t);
  uint32_t n_groups;
  uint32_t g = plan_scan(cnt, wt, &n_groups);
  for (int t = lo; t < hi; ++t)
    if (starts(t)) t0_list[g++] = t;
  __syncthreads();

  const int G = static_cast<int>(n_groups);
  const int pg = (G + kPlanThreads - 1) / kPlanThreads;
  const int glo = min(static_cast<int>(threadIdx.x) * pg, G), ghi = min(glo + pg, G);
  uint32_t tiles_sum = 0;
  bool bad = false;
  for (int gi = glo; gi < ghi; ++gi) {
    const int t0 = t0_list[gi], t1 = gi + 1 < G ? t0_list[gi + 1] : n_q;
    int b = __ldg(bid + t0);
    if (b < 0 || b >= n_req) { bad = true; b = b < 0 ? 0 : n_req - 1; }
    int pmax = -1;
    for (int t = t0; t < t1; ++t) pmax = max(pmax, __ldg(pos + t));
    if (pmax >= max_ctx) { bad = true; pmax = max_ctx - 1; }
    groups[gi] = make_int4(t0, t1 - t0, b, pmax);
    tiles_sum += group_tiles(pmax);
  }
  if (bad) report_device_error(kErrBadIndex);
  // Tile prefix per group: the indexer hands each CTA an equal, contiguous range of the
  // concatenated tile sequence (all groups, in order).
  uint32_t total_tiles;
  uint32_t ts = plan_scan(tiles_sum, wt, &total_tiles);
  for (int gi = glo; gi < ghi; ++gi) {
    unit_start[gi] = static_cast<int32_t>(ts);
    ts += group_tiles(groups[gi].w);
  }
  if (threadIdx.x == 0) {
    unit_start[G] = static_cast<int32_t>(total_tiles);
    plan->total_tiles = static_cast<int>(total_tiles);
    plan->pad = 0;
    plan->n_groups = G;
    plan->error = 0;
  }
}

// Largest g < G with tile_start[g] <= t (tile_start non-decreasing, size G + 1).
__device__ __forceinline__ int find_group(const int32_t* __restrict__ tile_start, int G, int t) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(tile_start + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

struct Unit {
  int t0, count, b, pmax, tile_begin, tile_end;
};

// Next piece of this CTA's tile range [cur, t_hi): the part that falls in one group (a unit:
// that group's queries against a run of its key tiles). Every role walks the same sequence.
__device__ __forceinline__ bool next_unit(const int4* groups, const int32_t* tile_start, int G,
                                          int& g, int& cur, int t_hi, Unit& x) {
  if (cur >= t_hi) return false;
  while (g < G - 1 && __ldg(tile_start + g + 1) <= cur) ++g;   // also skips empty groups
  const int4 rec = __ldg(groups + g);
  const int base = __ldg(tile_start + g);
  x.t0 = rec.x; x.count = rec.y; x.b = rec.z; x.pmax = rec.w;
  x.tile_begin = cur - base;
  x.tile_end = min(t_hi, __ldg(tile_start + g + 1)) - base;
  cur = base + x.tile_end;
  return true;
}

struct KeyRows {
  const int32_t* cu;
  const int32_t* block_table;   // nullptr: contiguous
  int max_pages;
  int n_pages;                  // pages in the pool (paged mode)
  int64_t n_rows;
};

// Row of the first key of the 64-key sub-tile that starts at position s (s % 64 == 0 when
// paged). Out-of-range pages map to a row past the tensor, which TMA fills with zeros.
__device__ __forceinline__ int32_t subtile_row(const KeyRows& kr, int b, int s) {
  if (kr.block_table == nullptr) return __ldg(kr.cu + b) + s;
  const int pi = s / kPageRows;
  const int page = pi < kr.max_pages ? __ldg(kr.block_table + static_cast<int64_t>(b) * kr.max_pages + pi) : -1;
  if (page < 0 || page >= kr.n_pages) return static_cast<int32_t>(kr.n_rows);
  return page * kPageRows;
}

// Row of key s of request b (contiguous: cu[b] + s; paged: through the block table), or -1.
__device__ __forceinline__ int64_t key_row(const KeyRows& kr, int b, int s) {
  if (kr.block_table == nullptr) return static_cast<int64_t>(__ldg(kr.cu + b)) + s;
  const int pi = s / kPageRows;
  const int page = pi < kr.max_pages ? __ldg(kr.block_table + static_cast<int64_t>(b) * kr.max_pages + pi) : -1;
  if (page < 0 || page >= kr.n_pages) return -1;
  return static_cast<int64_t>(page) * kPageRows + s % kPageRows;
}

template <int HI, int DI, bool F8>
__global__ void __launch_bounds__(Shape<HI, DI, F8>::kThreads, 1)
indexer_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
               const float* __restrict__ w, const int32_t* __restrict__ pos, KeyRows kr,
               const Plan* __restrict__ plan, const int4* __restrict__ groups,
               const int32_t* __restrict__ unit_start, float* __restrict__ scores,
               int64_t stride, int max_ctx, int n_q, uint32_t* __restrict__ hist,
               const float* __restrict__ q_scale, const float* __restrict__ k_scale) {
  using S = Shape<HI, DI, F8>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const uint32_t warp = warp_id(), lane = lane_id();
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + S::kOffAbort);
  auto bar = [&](int i) { return sbase + S::kOffBar + 8u * static_cast<uint32_t>(i); };
  // barrier indices
  const int kAFull = 0, kAEmpty = S::kStages, kBFull = 2 * S::kStages, kBEmpty = kBFull + 1,
            kAccFull = kBFull + 2, kAccEmpty = kBFull + 4, kWFull = kBFull + 6,
            kWEmpty = kBFull + 8;

  if ((sbase & 1023u) != 0) {                          // swizzle atoms need 1 KB alignment
    if (threadIdx.x == 0) report_device_error(kErrBadIndex | 0xA1u);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < S::kStages; ++i) { mbar_init(bar(kAFull + i), 1); mbar_init(bar(kAEmpty + i), 1); }
    mbar_init(bar(kBFull), 1);
    mbar_init(bar(kBEmpty), 1);
    for (int h = 0; h < 2; ++h) {
      mbar_init(bar(kAccFull + h), 1);
      mbar_init(bar(kAccEmpty + h), 4);
      mbar_init(bar(kWFull + h), 128);
      mbar_init(bar(kWEmpty + h), 128);
    }
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc<512>(sbase + S::kOffTmem);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + S::kOffTmem);
  // This CTA's share of the concatenated tile sequence: an equal contiguous range.
  const int n_tiles = plan->total_tiles, n_groups = plan->n_groups;
  const int t_lo = static_cast<int>(static_cast<int64_t>(n_tiles) * blockIdx.x / gridDim.x);
  const int t_hi = static_cast<int>(static_cast<int64_t>(n_tiles) * (blockIdx.x + 1) / gridDim.x);
  const int g_lo = t_lo < t_hi ? find_group(unit_start, n_groups, t_lo) : 0;

  if (warp == 8) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_q);
      int stage = 0;
      uint32_t phase = 0, b_uses = 0;
      int ug = g_lo, ucur = t_lo;
      Unit un;
      while (next_unit(groups, unit_start, n_groups, ug, ucur, t_hi, un)) {
        if (!mbar_wait(bar(kBEmpty), (b_uses & 1u) ^ 1u, 0x01, abort_flag)) break;
        ++b_uses;
        mbar_expect_tx(bar(kBFull), S::kBBytes);
        for (int a = 0; a < S::kAtoms; ++a)
          for (int hh = 0; hh < S::kBRows / 256; ++hh)
            tma_load_2d(sbase + S::kOffB + a * S::kBAtom + hh * 256 * S::kAtomBytes, &tm_q,
                        a * S::kAtomElems, un.t0 * HI + hh * 256, bar(kBFull));
        bool ok = true;
        for (int tile = un.tile_begin; tile < un.tile_end; ++tile) {
          if (!mbar_wait(bar(kAEmpty + stage), phase ^ 1u, 0x02, abort_flag)) { ok = false; break; }
          mbar_expect_tx(bar(kAFull + stage), S::kAStage);
          const uint32_t dst = sbase + S::kOffA + stage * S::kAStage;
          for (int sub = 0; sub < kKeysPerTile / kPageRows; ++sub) {
            const int32_t row = subtile_row(kr, un.b, tile * kKeysPerTile + sub * kPageRows);
            for (int a = 0; a < S::kAtoms; ++a)
              tma_load_2d(dst + a * S::kAAtom + sub * kPageRows * S::kAtomBytes, &tm_k,
                          a * S::kAtomElems, row, bar(kAFull + stage));
          }
          if (++stage == S::kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, b_uses = 0, acc_uses[2] = {0u, 0u};
      int ug = g_lo, ucur = t_lo;
      Unit un;
      while (!*abort_flag && next_unit(groups, unit_start, n_groups, ug, ucur, t_hi, un)) {
        if (!mbar_wait(bar(kBFull), b_uses & 1u, 0x03, abort_flag)) break;
        ++b_uses;
        tc_fence_after();
        // A group of at most one accumulator's queries (the decode batch's, the ends of
        // requests) uses the two accumulators on alternate tiles, so that its next MMA overlaps
        // this tile's epilogue; a larger group has one half of its queries in each.
        const bool alt = un.count <= S::kQPA;
        int nq[2];
        uint32_t idesc[2];
        for (int h = 0; h < 2; ++h) {
          nq[h] = alt ? un.count : max(0, min(un.count - h * S::kQPA, S::kQPA));
          uint32_t n_cols = static_cast<uint32_t>(nq[h] * HI);
          n_cols = (n_cols + 15u) & ~15u;
          idesc[h] = F8 ? idesc_e4m3(128, n_cols < 16u ? 16u : n_cols)
                        : idesc_bf16(128, n_cols < 16u ? 16u : n_cols, 0, 0);
        }
        bool ok = true;
        for (int tile = un.tile_begin; tile < un.tile_end && ok; ++tile) {
          if (!mbar_wait(bar(kAFull + stage), phase, 0x04, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_base = sbase + S::kOffA + stage * S::kAStage;
          for (int h = 0; h < 2; ++h) {
            if (nq[h] == 0 || (alt && h != (tile & 1))) continue;
            if (!mbar_wait(bar(kAccEmpty + h), (acc_uses[h] & 1u) ^ 1u, 0x05, abort_flag)) { ok = false; break; }
            ++acc_uses[h];
            tc_fence_after();
            const uint32_t b_base =
                sbase + S::kOffB + (alt ? 0 : h) * S::kQPA * HI * S::kAtomBytes;
#pragma unroll
            for (int kk = 0; kk < S::kKSteps; ++kk) {
              const int a = kk / S::kStepsPerAtom, off = (kk % S::kStepsPerAtom) * 32;
              const uint64_t da = smem_desc(a_base + a * S::kAAtom + off, 16, S::kSBO, S::kSwz);
              const uint64_t db = smem_desc(b_base + a * S::kBAtom + off, 16, S::kSBO, S::kSwz);
              if constexpr (F8)
                umma_ss_f8(tmem + static_cast<uint32_t>(h * 256), da, db, idesc[h], kk > 0 ? 1u : 0u);
              else
                umma_ss(tmem + static_cast<uint32_t>(h * 256), da, db, idesc[h], kk > 0 ? 1u : 0u);
            }
            umma_commit(bar(kAccFull + h));
          }
          umma_commit(bar(kAEmpty + stage));          // key tile free once both MMAs finish
          if (++stage == S::kStages) { stage = 0; phase ^= 1u; }
        }
        umma_commit(bar(kBEmpty));                    // Q tile free once the unit's MMAs finish
        if (!ok) break;
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogues (warps 0-7)
    const int h = static_cast<int>(warp >> 2);        // accumulator / query half
    const uint32_t quad = warp & 3u;                  // TMEM lane quadrant
    const int row = static_cast<int>(quad * 32u + lane);  // key inside the tile
    const uint32_t t_acc = tmem + ((quad * 32u) << 16) + static_cast<uint32_t>(h * 256);
    float* sw = reinterpret_cast<float*>(smem + S::kOffW) + h * S::kQPA * HI;
    int* spos = reinterpret_cast<int*>(smem + S::kOffPos) + h * S::kQPA;
    uint32_t acc_uses = 0, w_uses = 0;
    int ug = g_lo, ucur = t_lo;
    Unit un;
    while (!*abort_flag && next_unit(groups, unit_start, n_groups, ug, ucur, t_hi, un)) {
      const bool alt = un.count <= S::kQPA;          // the MMA issuer's choice, as above
      const int nq = alt ? un.count : max(0, min(un.count - h * S::kQPA, S::kQPA));
      if (nq == 0) continue;
      const int tq0 = un.t0 + (alt ? 0 : h * S::kQPA);
      // alternating: this half's tiles are those of its parity
      const int t_first = un.tile_begin + ((un.tile_begin & 1) != h);
      // The half's four warps share w / pos in smem: wait until all 128 threads finished with
      // the previous unit's copy, write this unit's, wait until every thread has written.
      if (!warp_wait(bar(kWEmpty + h), (w_uses & 1u) ^ 1u, 0x07, abort_flag)) break;
      for (int i = static_cast<int>(quad * 32u + lane); i < S::kQPA * HI; i += 128) {
        const int q = i / HI;
        const int64_t wi = static_cast<int64_t>(tq0 + q) * HI + (i % HI);
        float wv = q < nq ? __ldg(w + wi) : 0.f;
        if constexpr (F8) wv = q < nq ? wv * __ldg(q_scale + wi) : 0.f;   // w[t,h] * sq[t,h]
        sw[i] = wv;
      }
      for (int q = static_cast<int>(quad * 32u + lane); q < S::kQPA; q += 128)
        spos[q] = q < nq ? __ldg(pos + tq0 + q) : -1;
      mbar_arrive(bar(kWFull + h));
      if (!warp_wait(bar(kWFull + h), w_uses & 1u, 0x08, abort_flag)) break;
      ++w_uses;
      bool ok = true;
      // one tile of this unit; two loops below, so that the loop over every tile of a full
      // group stays as it was
      auto one_tile = [&](int tile) -> bool {
        float ks = 1.f;
        if constexpr (F8) {
          // the key's scale, loaded before the accumulator wait so the load is off the epilogue's
          // path: I = sk[s] * sum_h (w sq) ReLU(q8 . k8) (sk > 0 leaves the ReLU)
          const int64_t r = key_row(kr, un.b, tile * kKeysPerTile + row);
          ks = (r >= 0 && r < kr.n_rows) ? __ldg(k_scale + r) : 0.f;
        }
        if (!warp_wait(bar(kAccFull + h), acc_uses & 1u, 0x06, abort_flag)) return false;
        ++acc_uses;
        tc_fence_after();
        // Four partial sums per query (heads h with h % 4 == 0, 1, 2, 3), held as two packed
        // pairs so that one two-wide FMA serves two heads: chains of HI / 4 dependent FMAs
        // instead of HI, added at the end.
        float2 accp[S::kQPA][2];
#pragma unroll
        for (int q = 0; q < S::kQPA; ++q) {
          accp[q][0] = make_float2(0.f, 0.f);
          accp[q][1] = make_float2(0.f, 0.f);
        }
        // 64 columns per TMEM round trip; w read four columns at a time (broadcast LDS.128)
        static_assert((S::kQPA * HI) % 64 == 0, "epilogue chunks");
#pragma unroll
        for (int c0 = 0; c0 < S::kQPA * HI; c0 += 64) {
          uint32_t v[64];
          tmem_ld32(t_acc + static_cast<uint32_t>(c0), *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
          tmem_ld32(t_acc + static_cast<uint32_t>(c0 + 32), *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 64; j += 4) {
            const int col = c0 + j, q = col / HI;
            const float4 w4 = *reinterpret_cast<const float4*>(sw + col);
            const float2 r01 = make_float2(fmaxf(__uint_as_float(v[j]), 0.f),
                                           fmaxf(__uint_as_float(v[j + 1]), 0.f));
            const float2 r23 = make_float2(fmaxf(__uint_as_float(v[j + 2]), 0.f),
                                           fmaxf(__uint_as_float(v[j + 3]), 0.f));
            accp[q][0] = __ffma2_rn(make_float2(w4.x, w4.y), r01, accp[q][0]);
            accp[q][1] = __ffma2_rn(make_float2(w4.z, w4.w), r23, accp[q][1]);
          }
        }
        float acc[S::kQPA];
#pragma unroll
        for (int q = 0; q < S::kQPA; ++q)
          acc[q] = (accp[q][0].x + accp[q][0].y) + (accp[q][1].x + accp[q][1].y);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kAccEmpty + h));
        const int s = tile * kKeysPerTile + row;
        if constexpr (F8) {
#pragma unroll
          for (int q = 0; q < S::kQPA; ++q) acc[q] *= ks;
        }
#pragma unroll
        for (int q = 0; q < S::kQPA; ++q) {
          if (q < nq && s <= spos[q] && s < max_ctx)
            scores[static_cast<int64_t>(tq0 + q) * stride + s] = acc[q];
        }
        if (hist != nullptr && (s % kHistSample) == 0) {
          // First-digit histogram of a sample of the written scores (one position in
          // kHistSample; the lanes whose key sits at such a position), for the top-k after.
#pragma unroll
          for (int q = 0; q < S::kQPA; ++q) {
            if (q < nq && s <= spos[q] && s < max_ctx)
              atomicAdd(hist + static_cast<int64_t>(tq0 + q) * kHistBins +
                            first_digit(order_key(acc[q])), 1u);
          }
        }
        return true;
      };
      if (alt) {
        for (int tile = t_first; tile < un.tile_end; tile += 2)
          if (!one_tile(tile)) { ok = false; break; }
      } else {
        for (int tile = un.tile_begin; tile < un.tile_end; ++tile)
          if (!one_tile(tile)) { ok = false; break; }
      }
      mbar_arrive(bar(kWEmpty + h));                  // done reading this unit's w / pos
      if (!ok) break;
    }
  }

  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc<512>(tmem);
  }
}

template <int HI, int DI, bool F8>
int launch_indexer(const void* q_idx, const float* w, const void* k_idx, int64_t n_kv_rows,
                   const int32_t* pos, const int32_t* bid, int64_t n_q, int n_req, int max_ctx,
                   const KeyRows& kr, float* scores, int64_t stride, Plan* plan, int4* groups,
                   int32_t* unit_start, int32_t* t0_list, int n_ctas, uint32_t* hist,
                   const float* q_scale, const float* k_scale, int skip_le, cudaStream_t stream) {
  using S = Shape<HI, DI, F8>;
  if (hist != nullptr)
    DSA_CHECK_CUDA(cudaMemsetAsync(hist, 0, static_cast<size_t>(n_q) * kHistBins * sizeof(uint32_t),
                                   stream));
  const int n_req_eff = kr.block_table ? n_req : n_req;
  indexer_plan_kernel<<<1, kPlanThreads, 0, stream>>>(pos, bid, static_cast<int>(n_q), n_req_eff,
                                                      max_ctx, S::kGQ, skip_le, plan, groups,
                                                      unit_start, t0_list);
  DSA_CHECK_CUDA(cudaGetLastError());
  CUtensorMap tk, tq;
  int rc = make_tmap_2d(&tk, S::kTmaType, k_idx, static_cast<uint64_t>(n_kv_rows), DI,
                        S::kRowBytes, S::kAtomElems, kPageRows, S::kTmaSwz);
  if (rc) return rc;
  rc = make_tmap_2d(&tq, S::kTmaType, q_idx, static_cast<uint64_t>(n_q * HI), DI, S::kRowBytes,
                    S::kAtomElems, 256, S::kTmaSwz);
  if (rc) return rc;
  DSA_CHECK_CUDA(cudaFuncSetAttribute(indexer_kernel<HI, DI, F8>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmem));
  indexer_kernel<HI, DI, F8><<<n_ctas, S::kThreads, S::kSmem, stream>>>(
      tk, tq, w, pos, kr, plan, groups, unit_start, scores, stride, max_ctx,
      static_cast<int>(n_q), hist, q_scale, k_scale);
  DSA_CHECK_CUDA(cudaGetLastError());
  return DSA_OK;
}

}  // namespace

size_t indexer_plan_bytes(int64_t n_q) { return PlanLayout(n_q).bytes; }

int indexer_scores(const void* q_idx, const float* w, const void* k_idx, int64_t n_kv_rows,
                   const int32_t* cu, const int32_t* pos, const int32_t* bid, int64_t n_q, int n_req,
                   int Hi, int Di, int max_ctx, const int32_t* block_table, int max_pages,
                   int page_size, float* scores, int64_t stride, void* ws, size_t ws_bytes,
                   uint32_t* hist, const float* q_scale, const float* k_scale, int skip_le,
                   cudaStream_t stream) {
  if (n_q < 0 || max_ctx < 1 || n_kv_rows < 0)
    return fail(DSA_ERR_INVALID, "indexer: need n_q >= 0, max_ctx >= 1, n_kv_rows >= 0");
  if (n_q == 0) return DSA_OK;
  if (!q_idx || !w || !k_idx || !pos || !bid || !scores)
    return fail(DSA_ERR_INVALID, "indexer: null pointer");
  if (!block_table && !cu) return fail(DSA_ERR_INVALID, "indexer: need cu or block_table");
  if (block_table && (page_size != kPageRows || max_pages < 1))
    return fail(DSA_ERR_UNSUPPORTED, "indexer: paged KV needs page_size 64 (got %d)", page_size);
  if (n_q > (1 << 24) || n_kv_rows >= (1ll << 31) || n_q * Hi >= (1ll << 31))
    return fail(DSA_ERR_UNSUPPORTED, "indexer: sizes beyond 32-bit TMA coordinates");
  if (stride < max_ctx) return fail(DSA_ERR_INVALID, "indexer: score stride < max_ctx");
  const PlanLayout L(n_q);
  if (!ws || ws_bytes < L.bytes)
    return fail(DSA_ERR_WORKSPACE, "indexer: workspace of %zu bytes < %zu", ws_bytes, L.bytes);
  uint8_t* base = static_cast<uint8_t*>(ws);
  Plan* plan = reinterpret_cast<Plan*>(base + L.plan_off);
  int4* groups = reinterpret_cast<int4*>(base + L.groups_off);
  int32_t* unit_start = reinterpret_cast<int32_t*>(base + L.unit_off);
  int32_t* t0_list = reinterpret_cast<int32_t*>(base + L.t0_off);

  const int n_ctas = num_sms_cached();
  KeyRows kr{cu, block_table, max_pages, 0, n_kv_rows};
  if (block_table) kr.n_pages = static_cast<int>(n_kv_rows / kPageRows);
  const bool f8 = q_scale != nullptr;
  if (f8 != (k_scale != nullptr))
    return fail(DSA_ERR_INVALID, "indexer: FP8 rows need both q_scale and k_scale");
  if (f8) {
    if (Hi == 64 && Di == 128)
      return launch_indexer<64, 128, true>(q_idx, w, k_idx, n_kv_rows, pos, bid, n_q, n_req,
                                           max_ctx, kr, scores, stride, plan, groups, unit_start,
                                           t0_list, n_ctas, hist, q_scale, k_scale, skip_le, stream);
    return fail(DSA_ERR_UNSUPPORTED, "indexer: FP8 (Hi, Di) = (%d, %d) not built; supported "
                                     "(64, 128)", Hi, Di);
  }
  if (Hi == 64 && Di == 128)
    return launch_indexer<64, 128, false>(q_idx, w, k_idx, n_kv_rows, pos, bid, n_q, n_req,
                                          max_ctx, kr, scores, stride, plan, groups, unit_start,
                                          t0_list, n_ctas, hist, nullptr, nullptr, skip_le,
                                          stream);
  if (Hi == 4 && Di == 32)
    return launch_indexer<4, 32, false>(q_idx, w, k_idx, n_kv_rows, pos, bid, n_q, n_req, max_ctx,
                                        kr, scores, stride, plan, groups, unit_start, t0_list,
                                        n_ctas, hist, nullptr, nullptr, skip_le, stream);
  return fail(DSA_ERR_UNSUPPORTED, "indexer: (Hi, Di) = (%d, %d) not built; supported (64, 128), "
                                   "(4, 32)", Hi, Di);
}

cudaError_t indexer_read_errors(uint32_t* flags) { return read_and_clear_device_error(flags); }

}  // namespace dsa
