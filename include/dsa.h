/*
 * dsa.h -- C ABI of the GB300 (sm_103a) DSA "score, select, sparse read" path.
 *
 * The path has two steps:
 *
 *  1. dsa_index_topk: a lightweight indexer scores every causal history
 *     position of every query from a paged index-key cache and keeps the Top-K
 *     positions.  score(t, s) = sum_j w[t][j] * ReLU(q_idx[t][j] . k_idx[s]),
 *     j over 64 index heads of dimension 128.  Scoring, head weighting and
 *     selection run in one fused kernel that reads the paged cache directly and
 *     writes back only the indices ("Optimizing Inference for Hybrid Attention
 *     LLMs: A Practical Guide to Day-0 Adaptation", §3.1 Indexer Fusion; "Day-0
 *     Inference Adaptation and Optimization for Hybrid Attention
 *     Architectures", §3 Optimization 1; "Day0 Inference Support and
 *     Performance Optimization for New-Architecture LLMs", §4 item 1).
 *
 *  2. dsa_sparse_mla: a sparse attention kernel gathers only the selected
 *     576-wide latent KV rows (512 latent + 64 rope) and computes softmax
 *     attention of every query head over them; values are the first 512 dims
 *     ("Day0 Inference Support and Performance Optimization for
 *     New-Architecture LLMs", §2 item 2 and §4 "Sparse attention reads by
 *     index"; "Day0 Inference Optimization for a New Hybrid Attention
 *     Architecture: A Full-Stack Deep Dive", operator fusion item 1).
 *
 * Conventions shared by every entry point
 *  - All tensor arguments are caller-owned DEVICE pointers, row-major, densely
 *    packed, 16-byte aligned (stated otherwise where a weaker rule holds).
 *    Sizes are element counts.  The library never allocates, frees or
 *    synchronises on these calls (dsa_get_error excepted); work is enqueued on
 *    `stream` (a cudaStream_t passed as void*, NULL = legacy default stream),
 *    so the calls can be captured in a CUDA graph.
 *  - Paged caches: logical position s of sequence b lives in physical row
 *    page_table[b * max_pages_per_seq + s / page_size] * page_size + s % page_size
 *    of a cache shaped [num_pages, page_size, row_width].
 *  - Queries: sequence b owns query rows cu_q[b] .. cu_q[b+1]-1, which are its
 *    LAST (cu_q[b+1]-cu_q[b]) positions: query row t of sequence b sits at
 *    position pos(t) = seq_lens[b] - (cu_q[b+1]-cu_q[b]) + (t - cu_q[b]) and may
 *    attend to positions 0 .. pos(t) (causal, current token included).
 *    Decode: one query per sequence at position seq_lens[b]-1.  Prefill of a
 *    chunk: the chunk's tokens are the last positions of the cached sequence.
 *  - Workspace: caller-owned device memory of at least the bytes reported by
 *    the matching *_workspace_size() call.  Its first 16 bytes hold a sticky
 *    device error word (and the wait limit of dsa_workspace_set_wait_limit):
 *    call dsa_workspace_init() once after allocating it.
 *    Kernels OR error bits into it; dsa_get_error() reads and clears it.
 *  - Return value: DSA_OK if the work was enqueued.  Argument problems found
 *    on the host return DSA_ERR_INVALID_ARG / DSA_ERR_UNSUPPORTED before any
 *    launch; a failed launch returns DSA_ERR_CUDA.  Problems found on the
 *    device (a page id outside [0, num_pages), an index outside 0..pos(t), a
 *    pipeline wait that ran out) are reported later by dsa_get_error().  On
 *    any error the outputs are unspecified.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DSA_OK = 0,
    DSA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size or count       */
    DSA_ERR_UNSUPPORTED = 2,  /* valid request this build does not implement      */
    DSA_ERR_CUDA = 3,         /* a CUDA runtime/driver call or launch failed      */
    DSA_ERR_BAD_PAGE = 4,     /* device: page-table entry outside [0, num_pages)  */
    DSA_ERR_BAD_INDEX = 5,    /* device: selected index outside 0..pos(t)         */
    DSA_ERR_TIMEOUT = 6       /* device: a bounded pipeline wait ran out          */
} dsa_status;

/* Index-path element type, shared by q_idx and k_idx.  MXFP8 is E4M3 with one
 * E8M0 scale byte per 32 consecutive elements ("Day-0 Inference Adaptation and
 * Optimization for Hybrid Attention Architectures", §4 Optimization 2).
 * MXFP8_QBF16: MXFP8 index keys with q_idx passed in bf16; the fused indexer
 * quantises q_idx itself with dsa_quant_mxfp8's rule (the same codes and
 * scales, so the same indices), which saves the separate quantisation launch
 * of the query ("Day-0 Inference Adaptation and Optimization for Hybrid
 * Attention Architectures", §3 Optimization 1, input preparation). */
typedef enum { DSA_IDX_BF16 = 0, DSA_IDX_MXFP8 = 1, DSA_IDX_MXFP8_QBF16 = 2 } dsa_idx_dtype;

/* Main KV cache element type.  FP8_ROWSCALE: the 512 latent dims are E4M3 with
 * one fp32 scale per row, the 64 rope dims stay bf16.  FP8_TILE128: the same
 * with one fp32 scale per tile of 128 latent dims (four per row), the
 * per-token-head-tile granularity of "Day-0 Inference Adaptation and
 * Optimization for Hybrid Attention Architectures", §4 Optimization 2. */
typedef enum { DSA_KV_BF16 = 0, DSA_KV_FP8_ROWSCALE = 1, DSA_KV_FP8_TILE128 = 2 } dsa_kv_dtype;

/* Fixed dimensions of this build. */
#define DSA_INDEX_HEADS 64
#define DSA_INDEX_DIM 128
#define DSA_LATENT_DIM 576
#define DSA_VALUE_DIM 512

/* Short human-readable name of a status code (static storage). */
const char *dsa_status_string(dsa_status s);

/* Launch-shape tuning knobs, read on every call (0 = automatic).  Names:
 * "indexer_cluster" (CTAs per cluster, power of two <= 16), "indexer_stages"
 * (shared-memory ring depth of the cluster indexers: 2, 4 or 6 where it fits;
 * an odd value is taken one lower, since two threads take alternate tiles),
 * "indexer_group" (query rows per cluster: 1, 2 or 4; the MXFP8 indexer takes
 * 1, 2 or 3, a forced 4 as 3, and chooses 3 only when forced), "mla_splits"
 * (key splits per query row), "mla_pair" (with 128
 * heads, run the two 64-head CTAs of a query as a cluster sharing every
 * gathered row: 1 yes, -1 or 0 no), "mla_stream_k" (64-head CTAs, one per SM, share
 * all (row, head group, key tile) units evenly instead of a split grid: 1 yes
 * where it applies, -1 or 0 no (the split grid, whose CTAs issue their even
 * and odd key tiles from two threads, measured faster); it needs the workspace
 * dsa_sparse_mla_workspace_size reports, and a
 * smaller workspace of the split grid's size keeps it off), "mla_dsplit"
 * (128 heads, bf16 cache: one CTA pair per query row and key split that
 * splits the 576 latent dims between its two CTAs, so that every selected
 * row is gathered once, and exchanges partial logits over distributed shared
 * memory: 1 yes, -1 no (two 64-head CTAs per query, "mla_pair" and
 * "mla_stream_k" then apply), 0 automatic = yes when the launch needs more
 * than one wave of CTAs), "topk_cluster", "indexer_order" (0: the indexers
 * take query rows longest first, so that the launch does not end on a long row
 * started late; -1: plain grid order, for measuring what the order buys),
 * "indexer_flat" (bf16 indexer: one CTA per SM scores an even share of the
 * 128-position tiles of all query rows, writes the rows' score keys and
 * top-digit counts to the workspace, and the CTA that completes a row selects
 * its Top-K: 1 yes where it applies (at most 512 query rows, rows of at most
 * 49152 positions, the workspace dsa_index_topk_workspace_size reports), -1
 * no, 0 automatic = yes when every query row is its own sequence and the
 * rows hold at least 3 * 2^20 positions in all).
 * Returns 0, or -1 for an unknown name.  Results do not depend on them. */
int dsa_set_tuning(const char *name, int value);

/* ---------------------------------------------------------------- workspace */

/* Bytes of workspace dsa_index_topk / dsa_index_scores / dsa_topk_from_scores
 * need: the 256-byte error block, plus, where the flat bf16 indexer applies
 * (see "indexer_flat"), T x 2048 histogram words, T tile counters and
 * T x max_pages_per_seq x page_size score keys of 4 bytes.  A workspace of
 * only the error block is accepted and keeps the flat indexer off.  The flat
 * indexer zeroes its counters and histograms itself (enqueued on the call's
 * stream), so the workspace may be shared with dsa_sparse_mla. */
size_t dsa_index_topk_workspace_size(int32_t B, int32_t T, int32_t K, int32_t max_pages_per_seq,
                                     int32_t page_size);

/* Bytes of workspace dsa_sparse_mla needs for T query rows of H heads with K
 * selected slots each: the error word plus the partial results of its key
 * splits (or of its stream-K CTAs, when that mode applies; a workspace of only
 * the split grid's size is accepted and keeps stream-K off). */
size_t dsa_sparse_mla_workspace_size(int32_t T, int32_t H, int32_t K);

/* Zero the error word of a workspace (enqueued on stream).  Call once after
 * allocation; dsa_get_error() clears it again after each read. */
dsa_status dsa_workspace_init(void *workspace, size_t workspace_bytes, void *stream);

/* Synchronise `stream`, read the workspace's device error word, clear it and
 * return the first error it records (DSA_OK if none).  Not for the hot path. */
dsa_status dsa_get_error(void *workspace, void *stream);

/* Test hook for the failure path (the source pages have no counterpart).
 * Every pipeline wait inside the kernels gives up after 200 ms, records
 * DSA_ERR_TIMEOUT in the workspace's error word, and the kernel then drains
 * its own copies and tensor-core work, frees its tensor memory and returns.
 * This call (enqueued on `stream`) makes the kernels that use this workspace
 * give up after `microseconds` instead, so that a test can make the waits run
 * out on purpose; 0 restores the 200 ms default.  The setting lives in the
 * workspace (word 2 of its error block): dsa_workspace_init resets it,
 * dsa_get_error does not. */
dsa_status dsa_workspace_set_wait_limit(void *workspace, uint32_t microseconds, void *stream);

/* ---------------------------------------------------------------- indexer */

/* Fused indexer + Top-K.
 *   q_idx        [T, 64, 128]  bf16 (BF16, MXFP8_QBF16), or e4m3 codes (MXFP8)
 *   q_idx_scale  [T, 64, 4]    e8m0 bytes, 4-byte aligned (MXFP8 only, else NULL)
 *   head_w       [T, 64]       fp32 per-head weights
 *   k_idx_cache  [num_pages, page_size, 128]  bf16, or e4m3 codes (MXFP8, MXFP8_QBF16)
 *   k_idx_scale  [num_pages, page_size, 4]    e8m0 bytes, 16-byte aligned (MXFP8, MXFP8_QBF16)
 *   page_table   [B, max_pages_per_seq] int32; seq_lens [B]; cu_q [B+1] int32
 *   indices      [T, K] int32 OUT: for every query row, the min(K, pos(t)+1)
 *                positions with the highest scores (ties: lower position
 *                first), ascending, followed by -1 padding.
 * page_size must be a multiple of 64; max_pages_per_seq * page_size bounds
 * every seq_lens[b].  The cluster kernel keeps the scores on chip; the flat
 * bf16 kernel (see "indexer_flat") passes 4-byte score keys through the
 * workspace, 4 bytes per position (L2-resident at decode sizes). */
dsa_status dsa_index_topk(const void *q_idx, const uint8_t *q_idx_scale, const float *head_w,
                          const void *k_idx_cache, const uint8_t *k_idx_scale, int64_t num_pages,
                          const int32_t *page_table, int32_t max_pages_per_seq, const int32_t *seq_lens,
                          const int32_t *cu_q, int32_t B, int32_t T, int32_t K, int32_t page_size,
                          dsa_idx_dtype dtype, int32_t *indices, void *workspace, size_t workspace_bytes,
                          void *stream);

/* Test hook with the same arguments as dsa_index_topk that also writes the
 * fp32 scores: scores [T, ld_scores]; entry (t, s) for s <= pos(t) and
 * s < ld_scores, other entries untouched.  Same kernel, same selection. */
dsa_status dsa_index_scores(const void *q_idx, const uint8_t *q_idx_scale, const float *head_w,
                            const void *k_idx_cache, const uint8_t *k_idx_scale, int64_t num_pages,
                            const int32_t *page_table, int32_t max_pages_per_seq, const int32_t *seq_lens,
                            const int32_t *cu_q, int32_t B, int32_t T, int32_t K, int32_t page_size,
                            dsa_idx_dtype dtype, int32_t *indices, float *scores, int64_t ld_scores,
                            void *workspace, size_t workspace_bytes, void *stream);

/* Top-K of given fp32 score rows with the indexer's selection code: row r of
 * scores [R, ld] is valid on entries 0..lens[r]-1 (lens <= ld); out [R, K]
 * receives the selected positions as dsa_index_topk does.  Bit-exact
 * selection: the result depends only on the score values (-0 == +0). */
dsa_status dsa_topk_from_scores(const float *scores, int64_t ld, const int32_t *lens, int32_t R, int32_t K,
                                int32_t *out, void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------- sparse MLA */

/* Sparse MLA attention over the selected rows.
 *   q          [T, H, 576] bf16 query (latent 512 + rope 64)
 *   kv_cache   BF16: [num_pages, page_size, 576] bf16 latent rows
 *              FP8_ROWSCALE / FP8_TILE128: [num_pages, page_size, 512] e4m3
 *              latent dims
 *   kv_rope    FP8 only: [num_pages, page_size, 64] bf16 rope dims
 *   kv_scale   FP8_ROWSCALE: [num_pages, page_size] fp32 row scales;
 *              FP8_TILE128: [num_pages, page_size, 4] fp32, entry j scales
 *              latent dims 128j..128j+127
 *   indices    [T, K] int32 logical positions; entries < 0 are skipped
 *   out        [T, H, 512] bf16 OUT: sum_i softmax_i(scale * q_h . kv_i) kv_i[0:512]
 *   lse        [T, H] fp32 OUT (natural-log log-sum-exp of the scaled logits)
 *              or NULL.  A row with no valid index gets out = 0, lse = -inf.
 * H must be a multiple of 16 (at most 128). */
dsa_status dsa_sparse_mla(const void *q, const void *kv_cache, const void *kv_rope, const float *kv_scale,
                          int64_t num_pages, const int32_t *page_table, int32_t max_pages_per_seq,
                          const int32_t *seq_lens, const int32_t *cu_q, const int32_t *indices, int32_t B,
                          int32_t T, int32_t H, int32_t K, float scale, int32_t page_size, dsa_kv_dtype dtype,
                          void *out, float *lse, void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------- quantisers */

/* MXFP8 quantisation of n bf16 values (n a multiple of 32): every 32
 * consecutive values share one E8M0 scale 2^X with X = floor(log2(amax)) - 8
 * (clamped to [-127, 127]); elements are E4M3 of x / 2^X, round to nearest
 * even, saturating at +-448; an all-zero block gets scale byte 127 and zero
 * elements (OCP Microscaling v1.0; the index path's per-group-32 format of
 * "Day-0 Inference Adaptation and Optimization for Hybrid Attention
 * Architectures", §4 Optimization 2).
 *   x [n] bf16 in; q [n] e4m3 codes out; e8m0 [n/32] scale bytes out. */
dsa_status dsa_quant_mxfp8(const void *x, int64_t n, void *q, void *e8m0, void *stream);

/* FP8 quantisation of 576-wide latent rows: the 512 latent dims share one fp32
 * scale s = amax / 448 (1 when amax is 0), stored as E4M3(x / s) (round to
 * nearest even, saturating); the 64 rope dims are copied as bf16 ("Day0
 * Inference Adaptation and Performance Optimization for a Sparse Hybrid
 * Architecture LLM", §3.1, with one scale per row).
 *   kv [rows, 576] bf16 in; nope [rows, 512] e4m3, rope [rows, 64] bf16 and
 *   scale [rows] fp32 out. */
dsa_status dsa_quant_fp8_rows(const void *kv, int64_t rows, void *nope, void *rope, float *scale, void *stream);

/* As dsa_quant_fp8_rows with one scale per tile of 128 latent dims: tile j
 * (dims 128j..128j+127) has s_j = amax_j / 448 (1 when amax_j is 0) and
 * elements E4M3(x / s_j); the per-token-head-tile format of "Day-0 Inference
 * Adaptation and Optimization for Hybrid Attention Architectures", §4
 * Optimization 2 (and "Day0 Inference Support and Performance Optimization
 * for New-Architecture LLMs", §5 item 2).
 *   kv [rows, 576] bf16 in; nope [rows, 512] e4m3, rope [rows, 64] bf16 and
 *   scale [rows, 4] fp32 out. */
dsa_status dsa_quant_fp8_tiles(const void *kv, int64_t rows, void *nope, void *rope, float *scale, void *stream);

/* ---------------------------------------------------------------- cache append */

/* Writes new tokens' index keys and latent rows into their page slots,
 * quantised on the way to each cache's format: the per-token block formats
 * line up with the page layout, so nothing is staged ("Optimizing Inference
 * for Hybrid Attention LLMs: A Practical Guide to Day-0 Adaptation", §4
 * Hierarchical Quantization, key points 1-2).
 *   k_new      [T, 128] bf16 new index keys, or NULL (index cache untouched)
 *   kv_new     [T, 576] bf16 new latent rows, or NULL (KV cache untouched)
 *   page_table, max_pages_per_seq, seq_lens, cu_q, B: as for dsa_index_topk;
 *              seq_lens already counts the new tokens, and the new tokens of
 *              sequence b (cu_q[b]..cu_q[b+1]-1) are its last positions
 *   idx_dtype  BF16: k_cache [num_pages, page_size, 128] bf16, k_scale NULL;
 *              MXFP8: k_cache e4m3 codes, k_scale [num_pages, page_size, 4]
 *              e8m0 (dsa_quant_mxfp8's format)
 *   kv_dtype   BF16: kv_cache [num_pages, page_size, 576] bf16;
 *              FP8_ROWSCALE / FP8_TILE128: kv_cache [.., 512] e4m3, kv_rope
 *              [.., 64] bf16, kv_scale [num_pages, page_size] or [.., 4] fp32
 *              (dsa_quant_fp8_rows / dsa_quant_fp8_tiles formats)
 * Rows of other positions are not touched.  A token whose page id is out of
 * range, or whose position would be negative, writes nothing and is reported
 * through the workspace (DSA_ERR_BAD_PAGE / DSA_ERR_INVALID_ARG from
 * dsa_get_error).  The workspace needs at least 256 bytes (its error word). */
dsa_status dsa_cache_append(const void *k_new, const void *kv_new, const int32_t *page_table,
                            int32_t max_pages_per_seq, const int32_t *seq_lens, const int32_t *cu_q, int32_t B,
                            int32_t T, int32_t page_size, int64_t num_pages, dsa_idx_dtype idx_dtype, void *k_cache,
                            void *k_scale, dsa_kv_dtype kv_dtype, void *kv_cache, void *kv_rope, float *kv_scale,
                            void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------- no-allocation variant */

/* dsa_sparse_mla without a workspace, for callers that cannot allocate device
 * memory around the call (a latency-critical step that must not take the
 * synchronisation an allocation can imply, or a plug-in whose host framework
 * owns all device memory).  The source pages have no counterpart to this
 * call; it exists for such callers only.
 *   Arguments and results are those of dsa_sparse_mla (without workspace).
 *   Scratch: the split-K partials go to a fixed 32 MiB array in the library's
 *   device image, held by every GPU that loads the library until exit.  A
 *   request whose partials do not fit returns DSA_ERR_UNSUPPORTED.  The array
 *   holds the split grid's partials; stream-K (about 40 MB of partials on a
 *   GPU of ~150 SMs) therefore stays off here, with the same results.  The first
 *   call on a device looks the array's address up (cudaGetSymbolAddress);
 *   make it before any stream capture.  Every call on a device shares the
 *   array: calls whose kernels overlap on the GPU race and must not be issued.
 *   Device-side error bits go to the array's own error word, which each call
 *   clears; dsa_sparse_mla_static_get_error reads them back. */
dsa_status dsa_sparse_mla_static(const void *q, const void *kv_cache, const void *kv_rope, const float *kv_scale,
                                 int64_t num_pages, const int32_t *page_table, int32_t max_pages_per_seq,
                                 const int32_t *seq_lens, const int32_t *cu_q, const int32_t *indices, int32_t B,
                                 int32_t T, int32_t H, int32_t K, float scale, int32_t page_size, dsa_kv_dtype dtype,
                                 void *out, float *lse, void *stream);

/* The device-side errors of the last dsa_sparse_mla_static call on the current
 * device, as dsa_get_error reports them for a workspace: synchronises
 * `stream`, reads the static array's error word, clears it and returns the
 * first error it records (DSA_OK if none; DSA_ERR_CUDA if the array's address
 * cannot be looked up).  Not for the hot path. */
dsa_status dsa_sparse_mla_static_get_error(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
