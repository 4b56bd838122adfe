// kernels.h -- internal interface between the C ABI (dsa_abi.cu) and the
// kernel translation units.  Not installed; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace dsa {

// Fused indexer + Top-K (indexer_topk.cu).
struct IndexerArgs {
    const float *head_w;        // [T, 64]
    const uint8_t *q_scale;     // MXFP8: [T, 64, 4] e8m0
    const uint16_t *q_bf16;     // MXFP8 with the query quantised in the kernel: [T, 64, 128] bf16
    const uint8_t *k_scale;     // MXFP8: [rows, 4] e8m0
    const int32_t *page_table;  // [B, max_pages]
    const int32_t *seq_lens;    // [B]
    const int32_t *cu_q;        // [B+1]
    int32_t *indices;           // [T, K]
    float *scores;              // [T, ld_scores] (test hook) or null
    uint32_t *err;              // device error word
    int64_t num_pages;
    int64_t ld_scores;
    int32_t max_pages;
    int32_t B, T, K, page_size;
    int32_t stages;             // smem ring depth (<= 8)
    int32_t tiles_cap;          // 128-position tiles one CTA can hold keys for
    int32_t grid_order;         // 1: query rows in grid order instead of longest first (measurement knob)
    // flat kernel only (workspace buffers; hist and cnt zeroed before the launch)
    uint32_t *flat_keys;        // [T, ld_flat] order-preserving keys of the scores
    uint32_t *flat_hist;        // [T, indexer_flat_hist_bins()] top-digit histograms
    int32_t *flat_cnt;          // [T] tiles of the row scored so far
    int64_t ld_flat;            // keys per row (multiple of 4, >= max_pages * page_size)
    int32_t flat_cap_tiles;     // tiles one CTA may be given (multiple of 4)
};

struct TopkArgs {
    const float *scores;   // [R, ld]
    const int32_t *lens;   // [R]
    int32_t *out;          // [R, K]
    int64_t ld;
    int32_t R, K;
    int32_t chunk_cap;     // keys one CTA holds
};

size_t indexer_smem_bytes(int G, int stages, int tiles_cap);
size_t topk_smem_bytes(int chunk_cap);
cudaError_t launch_indexer_bf16(const CUtensorMap &tm_k, const CUtensorMap &tm_q, const IndexerArgs &a, int G,
                                int C, int groups, size_t smem, bool write_scores, cudaStream_t st);
cudaError_t launch_topk_from_scores(const TopkArgs &a, int C, size_t smem, cudaStream_t st);
// Clusters of C CTAs of the G-query indexer kernel with `smem` bytes that can
// be resident at once (0 if the shape cannot launch).
int indexer_max_active_clusters(int G, int C, size_t smem);
// Flat bf16 indexer: `ctas` CTAs (one per SM) share the 128-position tiles of
// all T query rows evenly; the CTA that completes a row selects its Top-K.
// Needs T <= indexer_flat_rows_max() and rows of at most
// indexer_flat_stage_keys(stages) positions.
int indexer_flat_rows_max();
int indexer_flat_hist_bins();  // per-row histogram words in the workspace
int indexer_flat_stage_keys(int stages);
size_t indexer_flat_smem_bytes(int stages, int T, int cap_tiles);
cudaError_t launch_indexer_flat(const CUtensorMap &tm_k, const CUtensorMap &tm_q, const IndexerArgs &a, int ctas,
                                size_t smem, cudaStream_t st);
// MXFP8 variant (G = 1 or 2 query rows of one sequence per cluster).
size_t indexer_mxfp8_smem_bytes(int G, int stages, int tiles_cap);
// quant_q: q_idx arrives in bf16 (a.q_bf16) and the kernel quantises it to
// MXFP8 itself (tm_q unused); otherwise tm_q maps the E4M3 codes and
// a.q_scale holds their scales.
cudaError_t launch_indexer_mxfp8(const CUtensorMap &tm_k, const CUtensorMap &tm_q, const IndexerArgs &a, int G, int C,
                                 int groups, size_t smem, bool write_scores, bool quant_q, cudaStream_t st);
int indexer_mxfp8_max_active_clusters(int G, int C, size_t smem);

// Sparse MLA (sparse_mla.cu).
struct MlaArgs {
    const uint16_t *q;          // [T, H, 576] bf16
    const uint8_t *kv;          // [num_pages*page_size, 576] bf16 rows, or [.., 512] E4M3 (FP8 rows)
    const uint8_t *kv_rope;     // FP8 rows: [num_pages*page_size, 64] bf16 rope dims
    const float *kv_scale;      // FP8 rows: [num_pages*page_size, kv_scales] fp32 scales
    int kv_scales;              // FP8: scales per row, 1 (one per row) or 4 (one per 128 latent dims)
    const int32_t *page_table;  // [B, max_pages]
    const int32_t *seq_lens;    // [B]
    const int32_t *cu_q;        // [B+1]
    const int32_t *indices;     // [T, K]
    uint16_t *out;              // [T, H, 512] bf16
    float *lse;                 // [T, H] or null
    float *part_o;              // [T, H/64, splits, 64, 512] fp32 partial outputs (splits > 1),
                                // or [2 * sk_ctas, 64, 512] in stream-K mode
    float *part_ml;             // the same slots x 2: running max (log2 domain) and sum
    uint32_t *err;
    int64_t num_pages;
    int32_t max_pages;
    int32_t B, T, H, K, page_size;
    int32_t splits;             // key splits per (query, head group)
    int32_t keys_per_split;     // multiple of the key tile
    // stream-K mode (sk_ctas > 0): each head group's sk_ctas / (H/64) CTAs
    // share its sk_units = T * sk_tpr (row, key tile) units evenly; CTA c of a
    // head group takes units [c U / Cg, (c+1) U / Cg), at most two rows
    int32_t sk_ctas, sk_tpr;
    int64_t sk_units;
    float scale_log2;           // softmax scale * log2(e)
    float scale;                // softmax scale
};

size_t mla_smem_bytes(int NH);
int mla_key_tile();
// NH = heads per CTA (16, 32 or 64; H must be a multiple).  tm_q: 2D map of
// q [T*H, 576] bf16, box 64 x NH, 128-byte swizzle.
// fp8: the cache holds E4M3 latent dims with one fp32 scale per row (kv,
// kv_rope, kv_scale), dequantised to bf16 on the way into shared memory.
// pair: with 128 heads, run the two 64-head CTAs of a query as a cluster that
// shares every gathered row.
// Workspace bytes of the split grid (host; the stream-K layout may need more).
size_t mla_split_workspace_size(int32_t T, int32_t H, int32_t K);
// Stream-K mode (a.sk_ctas > 0) needs NH = 64 and no pair.
cudaError_t launch_sparse_mla(const CUtensorMap &tm_q, const MlaArgs &a, int NH, bool fp8, bool pair,
                              cudaStream_t st);
// Merge the split partials of NH-head groups into out (and lse).
cudaError_t launch_mla_combine(const MlaArgs &a, int NH, cudaStream_t st);

// Sparse MLA for H = 128 with the latent dims split over a CTA pair
// (sparse_mla_ds.cu): bf16 cache, split grid (no stream-K), the split
// partial layout of launch_sparse_mla.
size_t mla_ds_smem_bytes();
cudaError_t launch_sparse_mla_ds(const MlaArgs &a, cudaStream_t st);

// Quantisers (quant.cu).
cudaError_t launch_quant_mxfp8(const uint16_t *x, int64_t n, uint8_t *q, uint8_t *e8m0, cudaStream_t st);
cudaError_t launch_quant_fp8_tiles(const uint16_t *kv, int64_t rows, uint8_t *nope, uint16_t *rope, float *scale,
                                   cudaStream_t st);

// Cache append: new tokens' index keys / latent rows into their page slots.
struct AppendArgs {
    const uint16_t *k_new;      // [T, 128] bf16 or null
    const uint16_t *kv_new;     // [T, 576] bf16 or null
    const int32_t *page_table;  // [B, max_pages]
    const int32_t *seq_lens;    // [B], counting the new tokens
    const int32_t *cu_q;        // [B + 1]: new tokens of sequence b are cu_q[b]..cu_q[b+1]-1
    int max_pages, B, page_size;
    int64_t T, num_pages;
    void *k_cache;              // [rows, 128] bf16 or e4m3 (null: not written)
    uint8_t *k_scale;           // MXFP8: [rows, 4] e8m0
    void *kv_cache;             // [rows, 576] bf16 or [rows, 512] e4m3 (null: not written)
    uint16_t *kv_rope;          // FP8: [rows, 64] bf16
    float *kv_scale;            // FP8: [rows] or [rows, 4] fp32
    uint32_t *err;              // workspace error word
};
// kv_scales: 0 bf16 latent rows, 1 FP8 with a row scale, 4 FP8 with tile scales.
cudaError_t launch_cache_append(const AppendArgs &a, bool idx_mxfp8, int kv_scales, cudaStream_t st);
cudaError_t launch_quant_fp8_rows(const uint16_t *kv, int64_t rows, uint8_t *nope, uint16_t *rope, float *scale,
                                  cudaStream_t st);

}  // namespace dsa
