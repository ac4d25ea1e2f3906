/*
 * dsa_rr.h — C ABI of the GB300 (sm_103a) round-robin sequence-shard DSA attention library.
 *
 * One shard of DeepSeek-V3.2-style sparse-attention prefill when tokens are dealt round robin
 * over `sp` sequence shards (flattened token g goes to shard g % sp):
 *
 *   dsa_rr_split_metadata  shard token list, batch ids, positions, shard cu_seqlens, row gather
 *   dsa_rr_split_decode_metadata  the same for a decode step's new tokens (positions continue
 *                          each request's context)
 *   dsa_rr_rerange         all-gathered (rank-major) KV rows -> logical token order
 *   dsa_rr_rerange_paged   the same rows straight into a paged KV cache (rerange + cache write)
 *   dsa_rr_cache_local_paged  a rank's own tokens only into its paged KV cache (the global KV
 *                          is dropped after attention)
 *   dsa_indexer_topk       lightning-indexer scores over the causal history + per-query top-k
 *     (= dsa_indexer_scores followed by dsa_topk_select, also exported on their own)
 *   dsa_sparse_mla         sparse MLA of every shard query over its top-k latent rows
 *
 * Conventions (every function):
 *   - Tensor pointers are DEVICE pointers owned by the caller; the library allocates no device
 *     memory. Scratch space comes from the caller (dsa_indexer_topk_workspace_size).
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = legacy default
 *     stream). Scalars are host values; no call reads device data back to the host, so the
 *     calls can be captured in a CUDA graph.
 *   - Return value: DSA_OK (0) or a negative DSA_ERR_* code; dsa_last_error_string() gives the
 *     reason (per host thread). Validation happens before anything is enqueued.
 *   - No exception, trap or device assert crosses this ABI. Kernels that meet an out-of-range
 *     index skip it and set a bit in a device error word (dsa_read_device_errors); every wait
 *     inside a kernel is bounded in time.
 *   - bf16 tensors are passed as `const void*` (IEEE bfloat16, little endian).
 *   - Row-major layouts; "[a, b]" lists dimensions outermost first. Rows of bf16 tensors handed
 *     to the tensor-core calls must start on 16-byte boundaries (the base pointer 16-byte
 *     aligned; row widths 2*Di and 2*dqk bytes are multiples of 16 for every supported shape).
 */
#ifndef DSA_RR_H
#define DSA_RR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dsa_stream_t; /* identical to cudaStream_t */

enum {
  DSA_OK = 0,
  DSA_ERR_INVALID = -1,     /* invalid argument (null pointer, negative size, rank >= sp ...) */
  DSA_ERR_UNSUPPORTED = -2, /* a shape the kernels are not built for */
  DSA_ERR_WORKSPACE = -3,   /* workspace missing or too small */
  DSA_ERR_CUDA = -4         /* a CUDA runtime / driver call failed (launch, tensor map ...) */
};

/* Bits of the device error word. */
#define DSA_DEVERR_TIMEOUT 0x80000000u    /* a bounded in-kernel wait gave up (low byte: site) */
#define DSA_DEVERR_BAD_INDEX 0x40000000u  /* an index input was out of range; it was skipped */
#define DSA_DEVERR_BAD_LENGTH 0x20000000u /* a query row exceeded max_ctx; the row was skipped */

/* Human-readable reason for the last non-zero return on this host thread. */
const char* dsa_last_error_string(void);

/* Library ABI version (increments on any signature change). */
int dsa_version(void);

/* Synchronise the device, OR every kernel's device error word into *flags and clear them. */
int dsa_read_device_errors(uint32_t* flags);

/*
 * Self-test of the bounded in-kernel wait (the pages have no counterpart: this checks the
 * library's failure detection). Enqueues one single-warp kernel that waits, with the same
 * bounded wait the tcgen05 kernels use, for an mbarrier phase that nothing completes. After
 * limit_cycles SM clock cycles (1 <= limit_cycles <= 2^40) the wait gives up, the kernel sets
 * DSA_DEVERR_TIMEOUT | 0xEE in the device error word and returns; dsa_read_device_errors then
 * reports it. Nothing faults, traps or hangs, and the CUDA context stays usable.
 * Errors: DSA_ERR_INVALID for a limit outside the range, DSA_ERR_CUDA for a failed launch.
 */
int dsa_selftest_bounded_wait(int64_t limit_cycles, dsa_stream_t stream);

/*
 * Measurement probe (no counterpart on the pages): the rate at which one SM brings selected
 * latent rows into shared memory, by either of the two mechanisms the sparse MLA could use for
 * its row gather ("[RFC]: Parallel strategy for Deepseek v3.2 like models", Pros: the MLA runs
 * all heads on the gathered rows). Enqueues n_ctas CTAs (one per SM at most); CTA i fills a
 * 3-slot ring of 48-row tiles in the MLA's 128B-swizzled layout from rows[i * n_tiles * 48 ..],
 * n_tiles tiles, with nothing consuming them, and writes the SM clock cycles its loop took to
 * cycles[i].
 *   c:     device, bf16 [n_rows, 576] (1,152-byte rows), 16-byte aligned; read only.
 *   rows:  device, int32 [n_ctas * n_tiles * 48], each in [0, n_rows) (others read row 0 and
 *          set DSA_DEVERR_BAD_INDEX).
 *   mode:  0 = 16-byte cp.async copies by three warps per slot (the MLA's path);
 *          1 = TMA tile::gather4 issued by `issuers` (1..32) lanes of one warp;
 *          2 = both at once: columns 0..511 by cp.async, 512..575 by tile::gather4;
 *          3 = no gather: CTA pairs (clusters of 2, n_ctas even) push 192 KB per round into
 *              each other's shared memory by bulk DSMEM copies, n_tiles rounds (the rate of
 *              the path the MLA's courier uses); rows and c are not read;
 *          4 = as 0 through registers (16-byte ld.global + st.shared);
 *          5 = columns 0..319 through registers, 320..575 by cp.async;
 *          6 = as 4 with every row of a warp in flight at once;
 *          7 = no gather: each tile is the 48 consecutive rows from its first listed row on,
 *              nine 64-column x 48-row TMA tiled boxes (rows past n_rows read zeros).
 *   cycles: device, uint64 [n_ctas], written.
 * Every in-kernel wait is bounded. Errors: DSA_ERR_INVALID for a null pointer, a size out of
 * range or a bad mode; DSA_ERR_CUDA for a failed launch.
 */
int dsa_probe_row_gather(const void* c, int64_t n_rows, const int32_t* rows, int n_ctas,
                         int n_tiles, int mode, int issuers, uint64_t* cycles,
                         dsa_stream_t stream);

/*
 * Host helper: number of tokens shard `rank` of `sp` holds, ceil((n_tokens - rank) / sp), or
 * 0 when rank >= n_tokens. Source: "[DeepSeek v3.2] 上下文并行详解", section 2.B
 * (arange(cp_rank, tokens, cp_size)). Returns -1 for sp < 1, rank < 0, rank >= sp or
 * n_tokens < 0.
 */
int64_t dsa_rr_shard_len(int64_t n_tokens, int sp, int rank);

/*
 * Round-robin split metadata for shard `rank` of `sp`, plus an optional row gather.
 * Source: "[DeepSeek v3.2] 上下文并行详解", section 2.B (nsa_cp_round_robin_split_data and the
 * metadata kernel that recomputes cu_seqlens and batch indices after the scatter) and section 4
 * part 1 (the "rank X token <-> batch Y position Z" mapping).
 *
 * Shard token t (0 <= t < n_r, n_r = dsa_rr_shard_len(n_tokens, sp, rank)) is the flattened
 * token g_t = rank + t*sp. Outputs (device, int32):
 *   cu_shard [n_req+1]  cu_shard[b] = number of shard tokens with g < cu[b]
 *   pos      [n_r]      g_t - cu[bid_t]           (position inside its request)
 *   bid      [n_r]      the largest b with cu[b] <= g_t (empty requests are skipped)
 *   gidx     [n_r]      g_t; may be NULL
 * Inputs: cu [n_req+1] int32 request offsets, cu[0] = 0, non-decreasing, cu[n_req] = n_tokens
 * (the caller guarantees this; it is not read back). n_req >= 1.
 * Row gather (optional): if src_rows != NULL, dst_rows[t, :] = src_rows[g_t, :] for rows of
 * row_bytes bytes (src [n_tokens, row_bytes], dst [n_r, row_bytes]); 16-byte vectors when both
 * pointers and row_bytes are multiples of 16, else byte copies.
 * Errors: DSA_ERR_INVALID for sp < 1, rank outside [0, sp), n_req < 1, n_tokens < 0 or a null
 * required pointer. n_tokens == 0 is valid (only cu_shard is written, all zeros).
 */
int dsa_rr_split_metadata(const int32_t* cu, int n_req, int64_t n_tokens, int sp, int rank,
                          int32_t* cu_shard, int32_t* pos, int32_t* bid, int32_t* gidx,
                          const void* src_rows, void* dst_rows, int64_t row_bytes,
                          dsa_stream_t stream);

/*
 * Round-robin split of a decode step's new tokens.
 * Source: "[RFC]: Parallel strategy for Deepseek v3.2 like models", "New proposal" (sequence
 * parallel over the token dimension for both prefill and decode); the dealing itself is the
 * prefill one ("[DeepSeek v3.2] 上下文并行详解", section 2.B). Reading: the flattened batch is
 * the step's new tokens, and a new token's position continues its request's context.
 *
 * Identical to dsa_rr_split_metadata over cu_new [n_req+1] (offsets of each request's new
 * tokens, cu_new[n_req] = n_tokens) except that
 *   pos[t] = pos_base[bid_t] + (g_t - cu_new[bid_t])
 * where pos_base [n_req] int32 device = the number of tokens of request b already in the KV
 * cache before this step. The outputs feed dsa_indexer_topk / dsa_sparse_mla with a block
 * table. Every argument is a device pointer or a host scalar, nothing is read back, so a decode
 * step built from these calls can be captured in a CUDA graph and replayed.
 * Errors: as dsa_rr_split_metadata; DSA_ERR_INVALID when pos_base is NULL.
 */
int dsa_rr_split_decode_metadata(const int32_t* cu_new, const int32_t* pos_base, int n_req,
                                 int64_t n_tokens, int sp, int rank, int32_t* cu_shard,
                                 int32_t* pos, int32_t* bid, int32_t* gidx, const void* src_rows,
                                 void* dst_rows, int64_t row_bytes, dsa_stream_t stream);

/*
 * Rerange an all-gathered buffer to logical token order.
 * Source: "[DeepSeek v3.2] 上下文并行详解", section 2.C (cp_all_gather_rerange_output) and
 * section 4 part 3 step B (the gathered rows come rank by rank, T0,T4,T1,T5,...; the rerange
 * restores T0,T1,T2,... so that the top-k sees logically contiguous KV).
 *
 * out[g, :] = gathered[off[g % sp] + g / sp, :] for 0 <= g < n_tokens, rows of row_bytes bytes.
 * off[q] = q * rank_stride_rows when rank_stride_rows > 0 (equal-size all-gather with padding,
 * rank_stride_rows >= ceil(n_tokens / sp)); rank_stride_rows == 0 means packed blocks,
 * off[q] = sum of the shard lengths of ranks < q.
 * gathered: [sp * rank_stride_rows or n_tokens, row_bytes]; out: [n_tokens, row_bytes]; the two
 * must not overlap. Errors: DSA_ERR_INVALID for sp < 1, a stride smaller than ceil(N/sp),
 * n_tokens < 0, row_bytes <= 0 or null pointers (n_tokens == 0 is a no-op).
 */
int dsa_rr_rerange(const void* gathered, void* out, int64_t n_tokens, int sp,
                   int64_t rank_stride_rows, int64_t row_bytes, dsa_stream_t stream);

/*
 * dsa_rr_rerange of several tensors that share the all-gather layout (the k_idx rows and the
 * latent rows of the same tokens), in one launch: for q < n_tensors,
 *   out[q][g, :] = gathered[q][off[g % sp] + g / sp, :]   (rows of row_bytes[q] bytes),
 * off[] as in dsa_rr_rerange. gathered / out / row_bytes are HOST arrays of n_tensors device
 * pointers and sizes (1 <= n_tensors <= 4); every buffer 16-byte aligned and every row_bytes a
 * multiple of 16. Same source passage as dsa_rr_rerange.
 * Errors: DSA_ERR_INVALID for a bad count, null or unaligned buffers, sp < 1, n_tokens < 0 or a
 * short stride; DSA_ERR_UNSUPPORTED above 2^31 16-byte chunks in total.
 */
int dsa_rr_rerange_multi(const void* const* gathered, void* const* out, const int64_t* row_bytes,
                         int n_tensors, int64_t n_tokens, int sp, int64_t rank_stride_rows,
                         dsa_stream_t stream);

/*
 * Rerange fused with the write of a paged KV cache.
 * Source: "[RFC]: Parallel strategy for Deepseek v3.2 like models", "New proposal" (the KV is
 * all-gathered before the KV-cache update step) and "[DeepSeek v3.2] 上下文并行详解", section 4
 * part 3 step B (rank-major gathered rows back to logical order). Reading: the two steps are
 * one pass, so the logical rows never exist as a separate buffer.
 *
 * For every logical token g < n_tokens with request b (the largest b with cu[b] <= g) and
 * position s = g - cu[b]:
 *   pool[block_table[b * max_pages + s / page_size] * page_size + s % page_size, :] =
 *       gathered[off[g % sp] + g / sp, :]
 * with off[] as in dsa_rr_rerange (rank_stride_rows > 0: padded blocks; 0: packed). Rows of
 * row_bytes bytes. cu [n_req+1] int32 device (cu[0] = 0, non-decreasing, cu[n_req] =
 * n_tokens); block_table [n_req, max_pages] int32 device; pool [pool_rows, row_bytes] device,
 * caller-owned; pool rows that no token maps to are not written. A token whose page entry is
 * negative, beyond max_pages or outside the pool is skipped and sets DSA_DEVERR_BAD_INDEX.
 * 16-byte vectors when both buffers and row_bytes are multiples of 16, else byte copies.
 * Errors: DSA_ERR_INVALID for sp < 1, n_tokens < 0 or >= 2^31, row_bytes <= 0, n_req < 1,
 * page_size < 1, max_pages < 1, a stride smaller than ceil(n_tokens / sp) or null pointers.
 */
int dsa_rr_rerange_paged(const void* gathered, void* pool, int64_t pool_rows, int64_t n_tokens,
                         int sp, int64_t rank_stride_rows, int64_t row_bytes, const int32_t* cu,
                         int n_req, const int32_t* block_table, int max_pages, int page_size,
                         dsa_stream_t stream);

/*
 * Keep only this rank's own tokens in its paged KV cache.
 * Source: "[DeepSeek v3.2] 上下文并行详解", section 4 part 3 step D: after attention the global
 * KV is not kept; the rank's KV-cache manager stores only the tokens it is responsible for (CP=4,
 * rank 1 keeps K1 and K5) in the cache pool, for the decode steps that follow.
 *
 * Shard token t (0 <= t < n_r = dsa_rr_shard_len(n_tokens, sp, rank)) is the flattened token
 * g_t = rank + t*sp of request b (the largest b with cu[b] <= g_t); its slot in the rank's cache
 * of request b is j = t - cu_shard[b], its index among request b's tokens on this rank
 * (cu_shard[b] = the number of shard tokens with g < cu[b]). Then
 *   pool[block_table[b * max_pages + j / page_size] * page_size + j % page_size, :] =
 *       local_rows[t, :]
 * local_rows [n_r, row_bytes] device: the rank's own rows in shard order (the rows its split
 * gathered, or block `rank` of a packed all-gather). cu [n_req+1] int32 device (cu[0] = 0,
 * non-decreasing, cu[n_req] = n_tokens); block_table [n_req, max_pages] int32 device, this
 * rank's pages (request b needs cu_shard[b+1] - cu_shard[b] slots); pool [pool_rows, row_bytes]
 * device; pool rows no token maps to are not written. A token whose page entry is negative,
 * beyond max_pages or outside the pool is skipped and sets DSA_DEVERR_BAD_INDEX. 16-byte vectors
 * when both buffers and row_bytes are multiples of 16, else byte copies.
 * Errors: DSA_ERR_INVALID for sp < 1, rank outside [0, sp), n_tokens < 0 or >= 2^31,
 * row_bytes <= 0, n_req < 1, page_size < 1, max_pages < 1 or null pointers (an empty shard is a
 * no-op).
 */
int dsa_rr_cache_local_paged(const void* local_rows, void* pool, int64_t pool_rows,
                             int64_t n_tokens, int sp, int rank, int64_t row_bytes,
                             const int32_t* cu, int n_req, const int32_t* block_table,
                             int max_pages, int page_size, dsa_stream_t stream);

/*
 * Bytes of scratch dsa_indexer_topk needs: the fp32 score rows [n_q, stride(max_ctx)] plus a
 * small scheduling area. max_ctx = an upper bound of pos_t + 1 over the queries.
 */
size_t dsa_indexer_topk_workspace_size(int64_t n_q, int max_ctx, int k);

/* Row stride (in floats) of the score rows for a given max_ctx (a multiple of 4). */
int64_t dsa_score_row_stride(int max_ctx);

/*
 * Lightning-indexer scores over each query's causal history (tcgen05 tensor cores).
 * The pages name this scan the bottleneck ("[RFC]: Parallel strategy for Deepseek v3.2 like
 * models", the comments on the indexer) but print no formula; the DeepSeek-V3.2 lightning
 * indexer defines, for shard query t of request b_t at position pos_t,
 *
 *     I[t, s] = sum_h w[t, h] * ReLU( sum_d q_idx[t, h, d] * k_idx[row(b_t, s), d] ),
 *     0 <= s <= pos_t,
 *
 * with row(b, s) = cu[b] + s (contiguous, logical order after the rerange) or
 * block_table[b * max_pages + s / page_size] * page_size + s % page_size (paged).
 *
 *   q_idx  bf16 [n_q, Hi, Di]     w fp32 [n_q, Hi]     k_idx bf16 [n_kv_rows, Di]
 *   cu     int32 [n_req+1] (contiguous mode; ignored when block_table != NULL)
 *   n_req  number of requests (rows of block_table when paged); bid must lie in [0, n_req)
 *   pos, bid int32 [n_q]          queries of one request must be consecutive in this order
 *   scores fp32 [n_q, score_stride]: row t receives I[t, 0..pos_t]; the rest is not written.
 * Supported: (Hi, Di) in {(64, 128), (4, 32)}; page_size 64 when paged. max_ctx >= pos_t + 1
 * for every t (rows that violate it are skipped and flagged DSA_DEVERR_BAD_LENGTH).
 * `workspace`/`workspace_bytes`: at least dsa_indexer_topk_workspace_size(n_q, max_ctx, 1)
 * bytes (only the scheduling area is used when scores are supplied separately).
 */
int dsa_indexer_scores(const void* q_idx, const float* w, const void* k_idx, int64_t n_kv_rows,
                       const int32_t* cu, int n_req, const int32_t* pos, const int32_t* bid,
                       int64_t n_q, int Hi, int Di, int max_ctx, const int32_t* block_table,
                       int max_pages, int page_size, float* scores, int64_t score_stride,
                       void* workspace, size_t workspace_bytes, dsa_stream_t stream);

/*
 * Per-query top-k of fp32 score rows ("history top-K", [RFC] page, comments): for row t of
 * length L_t = pos_t + 1 (scores[t * score_stride + s], 0 <= s < L_t), the k indices with the
 * largest score; equal scores go to the lower index; -0.0 equals +0.0; if L_t <= k all indices
 * are taken. topk [n_q, k] int32 lists the chosen indices in ascending order, padded with -1.
 * Scores must not be NaN. Radix select on CUDA cores.
 */
int dsa_topk_select(const float* scores, int64_t score_stride, const int32_t* pos, int64_t n_q,
                    int k, int max_ctx, int32_t* topk, dsa_stream_t stream);

/*
 * dsa_indexer_scores followed by dsa_topk_select, the score rows living in `workspace`.
 * topk: int32 [n_q, k], entries are positions s inside the query's request (0..pos_t) or -1.
 * A query whose history holds at most k keys (pos_t + 1 <= k) takes every key whatever its
 * scores, so the indexer leaves out every group of consecutive queries (one request, at most 8)
 * in which all queries are such; their score rows in the workspace are not written.
 * When max_ctx > 8192 the two steps are fused (same result): the indexer also counts, per
 * query, the first radix digit (top 11 bits of the order-preserving key) of one score in 16, the
 * top-k picks from those counts a threshold bin that very likely keeps at least k and only a few
 * thousand entries, reads each row once keeping exactly the entries at or above it, and selects
 * from that short list (rows where the sample misled are re-read in full). The workspace then
 * also holds these counts (dsa_indexer_topk_workspace_size includes them).
 */
int dsa_indexer_topk(const void* q_idx, const float* w, const void* k_idx, int64_t n_kv_rows,
                     const int32_t* cu, int n_req, const int32_t* pos, const int32_t* bid,
                     int64_t n_q, int Hi, int Di, int k, int max_ctx, const int32_t* block_table,
                     int max_pages, int page_size, int32_t* topk, void* workspace,
                     size_t workspace_bytes, dsa_stream_t stream);

/*
 * FP8 (E4M3) rows for the indexer ("[DeepSeek v3.2] 上下文并行详解", section 1: the round-robin
 * split is what allows an FP8 KV cache). The page names no format; the library reads it as:
 * E4M3 codes (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; largest finite 448;
 * S.1111.111 is NaN) with one fp32 scale per row of 128 values, the row standing for
 * code * scale. Quantisation: scale = amax / 448 (1 for a row of zeros), code = E4M3(x / scale)
 * rounded to nearest even and saturated at +-448, both divisions IEEE fp32.
 *
 * dsa_quantize_fp8_rows: x bf16 [rows, cols] -> codes uint8 [rows, cols], scales fp32 [rows];
 * cols must be 128 (DSA_ERR_UNSUPPORTED otherwise); x 8-byte and codes 4-byte aligned. Used
 * for k_idx (one row per token) and for q_idx (one row per (query, head): [n_q * Hi, 128]).
 */
int dsa_quantize_fp8_rows(const void* x, int64_t rows, int cols, void* codes, float* scales,
                          dsa_stream_t stream);

/*
 * FP8 latent (MLA) cache rows, the same reading per block of 128 latent values: a token's
 * 576-value latent row (512 latent + 64 rope values, bf16) is stored as a packed row of
 * DSA_FP8_LATENT_ROW_BYTES = 656 bytes: bytes [0, 512) the E4M3 codes of the 512 latent values,
 * [512, 528) four fp32 scales (value j uses scale j / 128), [528, 656) the 64 rope values,
 * bf16, unchanged. The attention consumes bf16 rows; a latent value expands to
 * bf16(fl32(code * scale)) (fp32 product, then bf16, both rounded to nearest even).
 * Packed rows are plain 656-byte rows for the split's row gather, the reranges and the paged
 * writes (the all-gathered cache moves in FP8).
 *
 * dsa_quantize_fp8_latent: c bf16 [rows, 576] -> packed uint8 [rows, 656].
 * dsa_dequantize_fp8_latent: packed uint8 [rows, 656] -> c bf16 [rows, 576].
 * Both device pointers 16-byte aligned, caller-owned; rows >= 0 (0: nothing to do).
 * Errors: DSA_ERR_INVALID for a null or misaligned pointer or rows < 0, DSA_ERR_CUDA for a
 * failed launch.
 */
#define DSA_FP8_LATENT_ROW_BYTES 656
int dsa_quantize_fp8_latent(const void* c, int64_t rows, void* packed, dsa_stream_t stream);
int dsa_dequantize_fp8_latent(const void* packed, int64_t rows, void* c, dsa_stream_t stream);

/*
 * Lightning-indexer scores on FP8 rows (tcgen05 kind::f8f6f4, fp32 accumulation): the indexer
 * of the dequantised rows,
 *     I[t, s] = sum_h w[t, h] * ReLU( (q_scale[t, h] q8[t, h, :]) . (k_scale[r] k8[r, :]) ),
 * r = row(b_t, s), computed as k_scale[r] * sum_h (w[t, h] q_scale[t, h]) ReLU(q8 . k8) (the
 * scales are positive). q8 uint8 E4M3 [n_q, Hi, Di], q_scale fp32 [n_q, Hi], k8 uint8 E4M3
 * [n_kv_rows, Di] (contiguous or a page pool), k_scale fp32 [n_kv_rows]. Every other argument,
 * the layouts, the workspace and the errors are those of dsa_indexer_scores / dsa_indexer_topk.
 * Supported: (Hi, Di) = (64, 128). Scales must be positive and finite.
 */
int dsa_indexer_scores_fp8(const void* q8, const float* q_scale, const float* w, const void* k8,
                           const float* k_scale, int64_t n_kv_rows, const int32_t* cu, int n_req,
                           const int32_t* pos, const int32_t* bid, int64_t n_q, int Hi, int Di,
                           int max_ctx, const int32_t* block_table, int max_pages, int page_size,
                           float* scores, int64_t score_stride, void* workspace,
                           size_t workspace_bytes, dsa_stream_t stream);
int dsa_indexer_topk_fp8(const void* q8, const float* q_scale, const float* w, const void* k8,
                         const float* k_scale, int64_t n_kv_rows, const int32_t* cu, int n_req,
                         const int32_t* pos, const int32_t* bid, int64_t n_q, int Hi, int Di,
                         int k, int max_ctx, const int32_t* block_table, int max_pages,
                         int page_size, int32_t* topk, void* workspace, size_t workspace_bytes,
                         dsa_stream_t stream);

/*
 * Sparse MLA on tcgen05 tensor cores (the selected rows are gathered into shared memory by
 * 16-byte cp.async copies for H = 128 and by TMA tile::gather4 for H = 8). "[RFC]: Parallel
 * strategy for Deepseek v3.2 like models": each query attends only its top-k keys, with all
 * heads at once. For query t and head h, over the valid entries of topk[t, :]:
 *
 *     S[h, j]   = scale * sum_{d < dqk} q[t, h, d] * c[row(b_t, idx_j), d]
 *     o[t, h,:] = sum_j softmax_j(S[h, :]) * c[row(b_t, idx_j), 0:dv]
 *     lse[t, h] = ln sum_j exp(S[h, j])
 *
 * (absorbed MLA: V is the first dv columns of the same latent row). An entry is valid when
 * 0 <= idx_j <= lim_t, lim_t = the last position of the query's request (contiguous mode:
 * cu[b+1] - cu[b] - 1) or of its block-table row (paged: max_pages * page_size - 1); -1 entries
 * are padding; an entry above lim_t is skipped (as if it were -1) and sets
 * DSA_DEVERR_BAD_INDEX. A query without valid entries gets o = 0 and lse = -inf.
 *   q  bf16 [n_q, H, dqk]     c bf16 [n_kv_rows, dqk]     topk int32 [n_q, k]
 *   cu int32 [n_req+1] (contiguous mode) / block_table int32 [n_req, max_pages] (paged)
 *   n_req >= 1; bid entries outside [0, n_req) read zero rows and set DSA_DEVERR_BAD_INDEX
 *   bid int32 [n_q]           o bf16 [n_q, H, dv]         lse fp32 [n_q, H] or NULL
 * Supported: (H, dqk, dv) in {(128, 576, 512), (8, 80, 64)}, page_size 64 when paged.
 * Softmax in fp32 (exp2 with a running maximum), P rounded to bf16 for the P.V product.
 * Index entries that land outside the KV buffer (a missing page) read zero rows and set
 * DSA_DEVERR_BAD_INDEX.
 */
int dsa_sparse_mla(const void* q, const void* c, int64_t n_kv_rows, const int32_t* cu, int n_req,
                   const int32_t* bid, const int32_t* topk, int64_t n_q, int H, int dqk, int dv,
                   int k, float scale, const int32_t* block_table, int max_pages, int page_size,
                   void* o, float* lse, dsa_stream_t stream);

/*
 * dsa_sparse_mla with a schedule for the persistent CTA pairs (H = 128 path). The pages have no
 * counterpart: this orders the work, the result is the same.
 *
 * Arguments and results are those of dsa_sparse_mla, plus pos (int32 [n_q], device): the query
 * positions, used only to estimate each query's work (a query at position p selects
 * min(p + 1, k) keys). Queries are sorted by that estimate, largest first, and dealt to the
 * pairs in rounds of alternating direction, so that the pairs finish together; o and lse are
 * bit-identical to dsa_sparse_mla's (each query's arithmetic does not depend on its pair).
 * With the positions given, an entry is valid only when it also lies in the query's causal
 * history: lim_t = min(pos_t, the request bound of dsa_sparse_mla); entries above it are
 * skipped and set DSA_DEVERR_BAD_INDEX.
 * workspace: device, 16-byte aligned, >= dsa_sparse_mla_workspace_size(n_q) bytes (the
 * schedule, int32 [n_q]); owned by the caller, not read before it is written. Errors as
 * dsa_sparse_mla, plus DSA_ERR_WORKSPACE for a short workspace and DSA_ERR_INVALID for a null
 * pos or a misaligned workspace. The (8, 80, 64) path checks the workspace but runs unscheduled.
 */
size_t dsa_sparse_mla_workspace_size(int64_t n_q);
int dsa_sparse_mla_balanced(const void* q, const void* c, int64_t n_kv_rows, const int32_t* cu,
                            int n_req, const int32_t* bid, const int32_t* pos,
                            const int32_t* topk, int64_t n_q, int H, int dqk, int dv, int k,
                            float scale, const int32_t* block_table, int max_pages,
                            int page_size, void* o, float* lse, void* workspace,
                            size_t workspace_bytes, dsa_stream_t stream);

/*
 * Allocation-free variant of dsa_indexer_topk. (The pages have no counterpart: this is a
 * convenience of the library, not a step of the method.)
 *
 * For callers that cannot allocate device memory -- a framework that reserved all device memory
 * in its own pool and forbids further cudaMalloc, a runtime without a CUDA allocator binding, or
 * a serving loop that must not call cudaMalloc / cudaFree because they can synchronise the
 * device. The scratch space lives in one file-scope __device__ array of
 * DSA_NOALLOC_SCRATCH_BYTES bytes that every GPU loading the library keeps until exit.
 * Arguments and results are those of dsa_indexer_topk without workspace / workspace_bytes.
 * The first call on a device (that device current) looks up the array's address with
 * cudaGetSymbolAddress and caches it per device; with lazy module loading that first call also
 * loads the library's device code on that device, which reserves the array and can synchronise
 * the device, so make it before any stream capture and outside latency-critical regions. The
 * cached address belongs to the device's current context: after cudaDeviceReset (or any
 * teardown of the primary context) it is stale, and the entry point must not be called again in
 * that process. All calls share the array: calls that may overlap on the GPU race and must not
 * be issued. Requests needing more scratch than the array (dsa_indexer_topk_workspace_size)
 * return DSA_ERR_WORKSPACE. No device memory is allocated or freed by the call itself.
 */
#define DSA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
int dsa_indexer_topk_noalloc(const void* q_idx, const float* w, const void* k_idx,
                             int64_t n_kv_rows, const int32_t* cu, int n_req, const int32_t* pos,
                             const int32_t* bid, int64_t n_q, int Hi, int Di, int k, int max_ctx,
                             const int32_t* block_table, int max_pages, int page_size,
                             int32_t* topk, dsa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_RR_H */
