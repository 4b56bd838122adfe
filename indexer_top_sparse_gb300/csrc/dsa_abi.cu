// dsa_abi.cu -- the C ABI declared in include/dsa.h: argument validation,
// TMA tensor-map encoding, launch-shape heuristics and the device error word.
// Every compute step runs in the kernels of indexer_topk.cu and sparse_mla.cu.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "dsa.h"
#include "kernels.h"

namespace {

using dsa::IndexerArgs;
using dsa::MlaArgs;
using dsa::TopkArgs;
using dsa::AppendArgs;

constexpr size_t kErrBytes = 256;  // error word block at the start of every workspace

// ---------------------------------------------------------------- tuning knobs
// 0 = automatic.  Set through dsa_set_tuning(); read on every call.
std::atomic<int> g_idx_cluster{0}, g_idx_stages{0}, g_idx_group{0}, g_mla_splits{0}, g_topk_cluster{0};
// 1: run the two 64-head CTAs of a 128-head query as a pair sharing each
// gathered row; -1: independent CTAs; 0: automatic (see mla_pair).
std::atomic<int> g_mla_pair{0};
// 1: stream-K sparse MLA whenever it applies; -1: never; 0: when the split
// grid would leave SMs idle (see mla_sk_ctas)
std::atomic<int> g_mla_sk{0};
// 1: 128-head bf16 sparse MLA on CTA pairs that split the latent dims
// (sparse_mla_ds.cu); -1: the 64-head kernels of sparse_mla.cu; 0: automatic
// (see mla_dsplit).
std::atomic<int> g_mla_ds{0};
// -1: the indexers take query rows in grid order; 0 (default): longest first
std::atomic<int> g_idx_order{0};
// 1: the flat bf16 indexer whenever it applies; -1: never; 0: for one query
// row per sequence (see plan_indexer_flat)
std::atomic<int> g_idx_flat{0};

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    return n;
}

size_t max_smem_optin() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 227 * 1024;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess || n <= 0)
        return 227 * 1024;
    return (size_t)n;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2D bf16 tensor [rows, cols] (row-major, dense) with box_rows x 64-column
// boxes and the 128-byte swizzle.
bool encode_2d_bf16(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn || rows == 0 || rows > (1ull << 31) || box_rows == 0 || box_rows > 256) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D uint8 tensor [rows, 128] (E4M3 codes) with 64-row x 128-byte boxes and the 128-byte swizzle.
bool encode_rows128_u8(CUtensorMap *m, const void *base, uint64_t rows) {
    auto fn = encode_fn();
    if (!fn || rows == 0 || rows > (1ull << 31)) return false;
    cuuint64_t dims[2] = {128, rows};
    cuuint64_t strides[1] = {128};
    cuuint32_t box[2] = {128, 64};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_rows128_bf16(CUtensorMap *m, const void *base, uint64_t rows) {
    return encode_2d_bf16(m, base, 128, rows, 64);
}

int mla_heads_per_cta(int H) {
    if (H == 16 || H == 32 || H == 64) return H;
    if (H % 64 == 0) return 64;
    return 0;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

struct IdxPlan {
    int G, C, stages, tiles_cap, groups;
    size_t smem;
};

// Resident clusters for a shape, cached per (device, G, C, smem).
int cached_max_clusters(int G, int C, size_t smem) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, size_t>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_tuple(dev, G, C, smem);
    {
        std::lock_guard<std::mutex> g(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    const int n = dsa::indexer_max_active_clusters(G, C, smem);
    std::lock_guard<std::mutex> g(mu);
    cache[key] = n;
    return n;
}

// Ring depth a forced "indexer_stages" value stands for in the cluster
// indexers: even (an odd value is taken one lower), since their two tcgen05
// issuing threads (and the MXFP8 kernel's two producers) take alternate
// tiles, and with an even depth every stage belongs to one of each -- each
// stage's barrier phases are then waited in order by one thread, so a parity
// wait cannot pass a phase early.
int even_stages(int forced) { return forced > 0 ? std::max(2, forced & ~1) : 0; }

// Launch shape of the fused indexer: G query rows per cluster, C CTAs per
// cluster, ring depth (even, see even_stages).  Preference: the fewest waves
// (clusters / resident clusters), then the most CTAs in flight, then the
// deepest ring; a CTA keeps at least 4 tiles of history unless the shape is
// forced.
bool plan_indexer(int B, int T, int max_len, IdxPlan *p) {
    const size_t smax = max_smem_optin();
    const int tiles_max = std::max(1, ceil_div(max_len, 128));
    const int g_force = g_idx_group.load(), c_force = g_idx_cluster.load(),
              s_force = even_stages(g_idx_stages.load());
    bool found = false;
    long long best_waves = 0, best_used = 0;
    int best_stages = 0;
    for (int G : {4, 2, 1}) {
        if (g_force ? G != g_force : (T <= B && G != 1)) continue;
        const int groups = G == 1 ? T : ceil_div(T, G) + B;
        for (int C = 1; C <= 16; C <<= 1) {
            if (c_force && C != c_force) continue;
            const int tiles_cap = ceil_div(tiles_max, C);
            if (!c_force && C > 1 && tiles_cap < 4) continue;
            for (int stages = 6; stages >= 2; stages -= 2) {
                if (s_force && stages != s_force) continue;
                size_t smem = dsa::indexer_smem_bytes(G, stages, tiles_cap);
                // TMEM: 2*64*G columns per CTA; cap the CTAs per SM through
                // shared memory so that allocations never wait on each other
                const int cols = std::max(128, 2 * 64 * G);
                const size_t floor_smem = (228u * 1024u) / (size_t)(512 / cols + 1) + 1;
                smem = std::max(smem, floor_smem);
                if (smem > smax) continue;
                const int resident = cached_max_clusters(G, C, smem);
                if (resident <= 0) continue;
                const long long waves = (groups + resident - 1) / resident;
                const long long used = (long long)std::min(groups, resident) * C;
                const bool better = !found || waves < best_waves ||
                                    (waves == best_waves && (used > best_used ||
                                                             (used == best_used && stages > best_stages)));
                if (better) {
                    *p = IdxPlan{G, C, stages, tiles_cap, groups, smem};
                    found = true;
                    best_waves = waves;
                    best_used = used;
                    best_stages = stages;
                }
            }
        }
        if (found) break;  // prefer the largest query group that fits
    }
    return found;
}

// The flat bf16 indexer (one CTA per SM sharing all rows' tiles evenly; the
// CTA that completes a row selects it): automatically for one query row per
// sequence (decode) with at least 3 * 2^20 positions in all, where streaming
// on every SM outweighs its fixed costs (a zeroing memset and a one-CTA
// selection per row after the last tile).  Measured on GB300, 32768-position
// rows: 96 rows 154 against 222 us, 160 rows 243 against 446 us (the cluster
// grid needs a second wave), 256 rows 374 against 470 us; below the
// threshold the cluster kernel was faster or equal (32 rows 72 against 60 us;
// 128 rows of 16384 positions 115 against 105 us).  Rows must fit the
// selection's staging (the query slots and the tile ring) and the row tables
// its shared memory.
struct FlatPlan {
    int ctas, stages, cap_tiles;
    size_t smem, zero_bytes, ws_bytes;  // workspace bytes past the error block (the first zero_bytes zeroed per call)
};

bool plan_indexer_flat(int B, int T, int max_len, FlatPlan *f) {
    const int forced = g_idx_flat.load();
    if (forced < 0 || T < 1 || T > dsa::indexer_flat_rows_max()) return false;
    if (forced == 0 && (T > B || g_idx_group.load() > 1 || g_idx_cluster.load() > 0 ||
                        (long long)T * max_len < (3LL << 20)))
        return false;
    const int ctas = sm_count();
    const long long tiles_max = std::max(1, ceil_div(max_len, 128));
    const long long cap = ((T * tiles_max + ctas - 1) / ctas + 1 + 3) & ~3LL;
    if (cap > 1024) return false;
    const size_t smax = max_smem_optin();
    const int s_force = g_idx_stages.load();
    for (int stages = 5; stages >= 3; --stages) {
        if (s_force && stages != s_force) continue;
        if (max_len > dsa::indexer_flat_stage_keys(stages)) break;  // fewer stages stage fewer keys
        const size_t smem = dsa::indexer_flat_smem_bytes(stages, T, (int)cap);
        if (smem > smax) continue;
        const size_t ld = (size_t)((max_len + 3) & ~3);
        const size_t zero = (size_t)T * dsa::indexer_flat_hist_bins() * 4 + (size_t)((T + 3) & ~3) * 4;
        *f = FlatPlan{ctas, stages, (int)cap, smem, zero, zero + (size_t)T * ld * 4};
        return true;
    }
    return false;
}

// Launch shape of the MXFP8 indexer: G query rows of one sequence per
// cluster (2 when a sequence has more query rows than there are sequences,
// i.e. prefill, if it fits; else 1), C CTAs per cluster, ring depth.
// Preference as for the bf16 indexer: the fewest waves, then the most CTAs in
// flight, then the deepest ring (even, see even_stages).
bool plan_indexer_mxfp8(int B, int T, int max_len, IdxPlan *p) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, size_t>, int> cache;
    const size_t smax = max_smem_optin();
    const int tiles_max = std::max(1, ceil_div(max_len, 128));
    // (a forced group of 4 takes this kernel's largest, 3)
    const int g_force = std::min(g_idx_group.load(), 3), c_force = g_idx_cluster.load(),
              s_force = even_stages(g_idx_stages.load());
    bool found = false;
    long long best_waves = 0, best_used = 0;
    int best_stages = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    for (int G : {3, 2, 1}) {
        if (g_force ? G != g_force : ((T <= B && G != 1) || G == 3)) continue;
        const int groups = G == 1 ? T : ceil_div(T, G) + B;
        for (int C = 1; C <= 16; C <<= 1) {
            if (c_force && C != c_force) continue;
            const int tiles_cap = ceil_div(tiles_max, C);
            if (!c_force && C > 1 && tiles_cap < 4) continue;
            for (int stages = 6; stages >= 2; stages -= 2) {
                if (s_force && stages != s_force) continue;
                const size_t smem = std::max(dsa::indexer_mxfp8_smem_bytes(G, stages, tiles_cap), (size_t)116 * 1024);
                if (smem > smax) continue;
                int resident;
                {
                    std::lock_guard<std::mutex> g(mu);
                    auto key = std::make_tuple(dev, G * 64 + C, stages, smem);
                    auto it = cache.find(key);
                    if (it == cache.end())
                        it = cache.emplace(key, dsa::indexer_mxfp8_max_active_clusters(G, C, smem)).first;
                    resident = it->second;
                }
                if (resident <= 0) continue;
                const long long waves = (groups + resident - 1) / resident;
                const long long used = (long long)std::min(groups, resident) * C;
                if (!found || waves < best_waves ||
                    (waves == best_waves && (used > best_used || (used == best_used && stages > best_stages)))) {
                    *p = IdxPlan{G, C, stages, tiles_cap, groups, smem};
                    found = true;
                    best_waves = waves;
                    best_used = used;
                    best_stages = stages;
                }
            }
        }
        if (found) break;  // prefer the larger query group when it fits
    }
    return found;
}

int mla_groups(int H) {
    const int nh = mla_heads_per_cta(H);
    return nh ? H / nh : 1;
}

int mla_splits(int T, int H, int K) {
    int forced = g_mla_splits.load();
    const int tile = dsa::mla_key_tile();
    const int max_splits = std::max(1, std::min(16, ceil_div(std::max(K, 1), tile)));
    const int min_splits = ceil_div(std::max(K, 1), 2048);  // a CTA resolves at most 2048 keys
    if (forced > 0) return std::max(min_splits, std::min(forced, max_splits));
    const long long pairs = (long long)T * mla_groups(H);
    const int nsm = sm_count();
    if (pairs >= nsm) return min_splits;
    return std::max(min_splits, std::min<int>(max_splits, (int)(nsm / pairs)));
}

// Pairs of 64-head CTAs that share every gathered row over distributed shared
// memory: only when asked for.  Each CTA of a pair may overwrite the rows it
// forwarded only after they have landed in the peer, and with that wait the
// pair measured slower than independent CTAs on GB300 (131k chunked FP8
// prefill: 221.5 against 216.2 ms of MLA; 32 x 32768 decode: 2 us slower).
// 128-head bf16 launches of more than one wave take the dims-split pair.
bool mla_pair(int T, int H, int splits) {
    (void)T;
    (void)splits;
    return g_mla_pair.load() > 0 && mla_heads_per_cta(H) == 64 && H == 128;
}

// Stream-K sparse MLA: CTAs (one per SM) for T rows of H heads with K keys,
// or 0 for the split grid.  It applies with 64-head CTAs when every CTA gets
// 2..tpr key tiles (so a CTA's run spans at most two (row, head group) pairs
// and its row table fits).  Only when asked for: the split grid issues each
// CTA's even and odd tiles from two threads, stream-K from one, and on GB300
// the split grid measured faster on both decode workloads (64 x 4k-128k FP8
// decode: 115.7 against 127.3 us; 32 x 32768 bf16 decode: 55.5 against
// 70.0 us).
int mla_sk_ctas(int T, int H, int K) {
    const int forced = g_mla_sk.load();
    if (forced <= 0 || mla_heads_per_cta(H) != 64 || g_mla_splits.load() > 0 || g_mla_pair.load() > 0 || T <= 0 ||
        K <= 0)
        return 0;
    const int nsm = sm_count(), tile = dsa::mla_key_tile(), tpr = ceil_div(K, tile);
    const int groups = mla_groups(H), cg = nsm / groups;  // CTAs per head group
    const long long units = (long long)T * tpr;           // per head group
    const long long per = (units + cg - 1) / cg;
    if (cg < 1 || units < 2LL * cg || per > tpr || per * tile > 2048) return 0;
    return cg * groups;
}
// The dims-split pair kernel (128 heads, bf16 cache) gathers each selected
// row once and runs M = 128 logits MMAs, but exchanges 32 KB of partial
// logits per 64-key tile over distributed shared memory.  Automatically when
// the launch takes more than one wave of CTAs, where it measured faster on
// GB300 (16k prefill: 19.8 against 24.9 ms); within one wave two independent
// 64-head CTAs per query are faster (32 x 32768 decode: 64.2 against 67.5 us).
bool mla_dsplit(int T, int H, bool fp8, int splits) {
    const int forced = g_mla_ds.load();
    if (forced < 0 || H != 128 || fp8) return false;
    return forced > 0 || 2LL * T * splits > sm_count();
}
size_t mla_sk_workspace(int ctas) { return kErrBytes + (size_t)2 * ctas * 64 * (512 + 2) * sizeof(float); }

__global__ void set_word_kernel(uint32_t *word, uint32_t value) { *word = value; }

dsa_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return DSA_OK;
    fprintf(stderr, "[dsa] CUDA error: %s\n", cudaGetErrorString(e));
    return DSA_ERR_CUDA;
}

dsa_status index_common(const void *q_idx, const uint8_t *q_idx_scale, const float *head_w, const void *k_idx_cache,
                        const uint8_t *k_idx_scale, int64_t num_pages, const int32_t *page_table,
                        int32_t max_pages_per_seq, const int32_t *seq_lens, const int32_t *cu_q, int32_t B,
                        int32_t T, int32_t K, int32_t page_size, dsa_idx_dtype dtype, int32_t *indices,
                        float *scores, int64_t ld_scores, void *workspace, size_t workspace_bytes, void *stream) {
    if (T < 0 || B < 1 || K < 1 || page_size < 1 || max_pages_per_seq < 1 || num_pages < 1) return DSA_ERR_INVALID_ARG;
    if (!q_idx || !head_w || !k_idx_cache || !page_table || !seq_lens || !cu_q || !indices || !workspace)
        return DSA_ERR_INVALID_ARG;
    if (!aligned16(q_idx) || !aligned16(k_idx_cache) || !aligned16(workspace)) return DSA_ERR_INVALID_ARG;
    // (the error block is the minimum; the flat indexer runs only in a
    // workspace of the size dsa_index_topk_workspace_size reports)
    if (workspace_bytes < kErrBytes) return DSA_ERR_INVALID_ARG;
    if (dtype != DSA_IDX_BF16 && dtype != DSA_IDX_MXFP8 && dtype != DSA_IDX_MXFP8_QBF16) return DSA_ERR_UNSUPPORTED;
    if (dtype == DSA_IDX_MXFP8 && (!q_idx_scale || !k_idx_scale || !aligned16(k_idx_scale) ||
                                   (reinterpret_cast<uintptr_t>(q_idx_scale) & 3u)))
        return DSA_ERR_INVALID_ARG;
    if (dtype == DSA_IDX_MXFP8_QBF16 && (q_idx_scale || !k_idx_scale || !aligned16(k_idx_scale)))
        return DSA_ERR_INVALID_ARG;
    if (page_size % 64 != 0) return DSA_ERR_UNSUPPORTED;
    if (T == 0) return DSA_OK;
    const long long max_len = (long long)max_pages_per_seq * page_size;
    if (max_len > (1LL << 30) || (long long)num_pages * page_size > (1LL << 31)) return DSA_ERR_UNSUPPORTED;
    if (dtype == DSA_IDX_MXFP8 || dtype == DSA_IDX_MXFP8_QBF16) {
        const bool quant_q = dtype == DSA_IDX_MXFP8_QBF16;
        IdxPlan plan;
        if (!plan_indexer_mxfp8(B, T, (int)max_len, &plan) || plan.groups > 65535) return DSA_ERR_UNSUPPORTED;
        CUtensorMap tk, tq;
        if (!encode_rows128_u8(&tk, k_idx_cache, (uint64_t)num_pages * page_size)) return DSA_ERR_CUDA;
        if (quant_q) tq = tk;  // unused: the kernel reads the bf16 query itself
        else if (!encode_rows128_u8(&tq, q_idx, (uint64_t)T * 64)) return DSA_ERR_CUDA;
        IndexerArgs a{};
        a.head_w = head_w;
        a.q_scale = quant_q ? nullptr : q_idx_scale;
        a.q_bf16 = quant_q ? static_cast<const uint16_t *>(q_idx) : nullptr;
        a.k_scale = k_idx_scale;
        a.page_table = page_table;
        a.seq_lens = seq_lens;
        a.cu_q = cu_q;
        a.indices = indices;
        a.scores = scores;
        a.err = reinterpret_cast<uint32_t *>(workspace);
        a.num_pages = num_pages;
        a.ld_scores = ld_scores;
        a.max_pages = max_pages_per_seq;
        a.B = B;
        a.T = T;
        a.K = K;
        a.page_size = page_size;
        a.stages = plan.stages;
        a.tiles_cap = plan.tiles_cap;
        a.grid_order = g_idx_order.load() < 0;
        return cuda_status(dsa::launch_indexer_mxfp8(tk, tq, a, plan.G, plan.C, plan.groups, plan.smem,
                                                     scores != nullptr, quant_q, static_cast<cudaStream_t>(stream)));
    }
    FlatPlan flat;
    const bool use_flat = !scores && plan_indexer_flat(B, T, (int)max_len, &flat) &&
                          workspace_bytes >= kErrBytes + flat.ws_bytes;
    IdxPlan plan{};
    if (!use_flat && (!plan_indexer(B, T, (int)max_len, &plan) || plan.groups > 65535)) return DSA_ERR_UNSUPPORTED;
    CUtensorMap tk, tq;
    if (!encode_rows128_bf16(&tk, k_idx_cache, (uint64_t)num_pages * page_size)) return DSA_ERR_CUDA;
    if (!encode_rows128_bf16(&tq, q_idx, (uint64_t)T * 64)) return DSA_ERR_CUDA;
    IndexerArgs a{};
    a.head_w = head_w;
    a.page_table = page_table;
    a.seq_lens = seq_lens;
    a.cu_q = cu_q;
    a.indices = indices;
    a.scores = scores;
    a.err = reinterpret_cast<uint32_t *>(workspace);
    a.num_pages = num_pages;
    a.ld_scores = ld_scores;
    a.max_pages = max_pages_per_seq;
    a.B = B;
    a.T = T;
    a.K = K;
    a.page_size = page_size;
    a.grid_order = g_idx_order.load() < 0;
    if (use_flat) {
        // workspace past the error block: [T][bins] histograms, [T] tile
        // counters (both zeroed here), [T][ld] keys
        uint8_t *base = static_cast<uint8_t *>(workspace) + kErrBytes;
        a.flat_hist = reinterpret_cast<uint32_t *>(base);
        a.flat_cnt = reinterpret_cast<int32_t *>(base + (size_t)T * dsa::indexer_flat_hist_bins() * 4);
        a.flat_keys = reinterpret_cast<uint32_t *>(base + flat.zero_bytes);
        a.ld_flat = (max_len + 3) & ~3LL;
        a.flat_cap_tiles = flat.cap_tiles;
        a.stages = flat.stages;
        cudaError_t e = cudaMemsetAsync(base, 0, flat.zero_bytes, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_status(e);
        return cuda_status(dsa::launch_indexer_flat(tk, tq, a, flat.ctas, flat.smem, static_cast<cudaStream_t>(stream)));
    }
    a.stages = plan.stages;
    a.tiles_cap = plan.tiles_cap;
    return cuda_status(dsa::launch_indexer_bf16(tk, tq, a, plan.G, plan.C, plan.groups, plan.smem,
                                                scores != nullptr, static_cast<cudaStream_t>(stream)));
}

size_t split_workspace_size(int32_t T, int32_t H, int32_t K) {
    if (T <= 0 || H <= 0 || K <= 0) return kErrBytes;
    const int splits = mla_splits(T, H, K);
    if (splits <= 1) return kErrBytes;
    const size_t rows = (size_t)T * mla_groups(H) * splits * 64;
    return kErrBytes + rows * 512 * sizeof(float) + rows * 2 * sizeof(float);
}

}  // namespace

namespace dsa {
size_t mla_split_workspace_size(int32_t T, int32_t H, int32_t K) { return split_workspace_size(T, H, K); }
}  // namespace dsa

extern "C" {

const char *dsa_status_string(dsa_status s) {
    switch (s) {
        case DSA_OK: return "ok";
        case DSA_ERR_INVALID_ARG: return "invalid argument";
        case DSA_ERR_UNSUPPORTED: return "unsupported";
        case DSA_ERR_CUDA: return "CUDA error";
        case DSA_ERR_BAD_PAGE: return "page id out of range";
        case DSA_ERR_BAD_INDEX: return "selected index out of range";
        case DSA_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown";
}

int dsa_set_tuning(const char *name, int value) {
    if (!name) return -1;
    if (!strcmp(name, "indexer_cluster")) g_idx_cluster = value;
    else if (!strcmp(name, "indexer_stages")) g_idx_stages = value;
    else if (!strcmp(name, "indexer_group")) g_idx_group = value;
    else if (!strcmp(name, "mla_splits")) g_mla_splits = value;
    else if (!strcmp(name, "mla_pair")) g_mla_pair = value;
    else if (!strcmp(name, "mla_stream_k")) g_mla_sk = value;
    else if (!strcmp(name, "mla_dsplit")) g_mla_ds = value;
    else if (!strcmp(name, "topk_cluster")) g_topk_cluster = value;
    else if (!strcmp(name, "indexer_order")) g_idx_order = value;
    else if (!strcmp(name, "indexer_flat")) g_idx_flat = value;
    else return -1;
    return 0;
}

size_t dsa_index_topk_workspace_size(int32_t B, int32_t T, int32_t K, int32_t max_pages_per_seq,
                                     int32_t page_size) {
    (void)K;
    FlatPlan flat;
    const long long max_len = (long long)max_pages_per_seq * page_size;
    if (B >= 1 && T >= 1 && max_len >= 1 && max_len <= (1LL << 30) && plan_indexer_flat(B, T, (int)max_len, &flat))
        return kErrBytes + flat.ws_bytes;
    return kErrBytes;
}

size_t dsa_sparse_mla_workspace_size(int32_t T, int32_t H, int32_t K) {
    const size_t split = split_workspace_size(T, H, K);
    const int sk = mla_sk_ctas(T, H, K);
    return sk > 0 ? std::max(split, mla_sk_workspace(sk)) : split;
}

dsa_status dsa_workspace_init(void *workspace, size_t workspace_bytes, void *stream) {
    if (!workspace || workspace_bytes < kErrBytes) return DSA_ERR_INVALID_ARG;
    return cuda_status(cudaMemsetAsync(workspace, 0, kErrBytes, static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_workspace_set_wait_limit(void *workspace, uint32_t microseconds, void *stream) {
    if (!workspace || !aligned16(workspace)) return DSA_ERR_INVALID_ARG;
    // one 4-byte write of word 2 of the error block, ordered on the stream
    set_word_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<uint32_t *>(workspace) + 2,
                                                                       microseconds);
    return cuda_status(cudaGetLastError());
}

dsa_status dsa_get_error(void *workspace, void *stream) {
    if (!workspace) return DSA_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t w[2] = {0, 0};
    cudaError_t e = cudaMemcpyAsync(w, workspace, sizeof w, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof w, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_status(e);
    for (int code = 1; code < 32; ++code)
        if (w[0] & (1u << code)) {
            if (code == DSA_ERR_TIMEOUT) fprintf(stderr, "[dsa] device wait timed out at site 0x%x\n", w[1]);
            return static_cast<dsa_status>(code);
        }
    return DSA_OK;
}

dsa_status dsa_index_topk(const void *q_idx, const uint8_t *q_idx_scale, const float *head_w,
                          const void *k_idx_cache, const uint8_t *k_idx_scale, int64_t num_pages,
                          const int32_t *page_table, int32_t max_pages_per_seq, const int32_t *seq_lens,
                          const int32_t *cu_q, int32_t B, int32_t T, int32_t K, int32_t page_size,
                          dsa_idx_dtype dtype, int32_t *indices, void *workspace, size_t workspace_bytes,
                          void *stream) {
    return index_common(q_idx, q_idx_scale, head_w, k_idx_cache, k_idx_scale, num_pages, page_table,
                        max_pages_per_seq, seq_lens, cu_q, B, T, K, page_size, dtype, indices, nullptr, 0,
                        workspace, workspace_bytes, stream);
}

dsa_status dsa_index_scores(const void *q_idx, const uint8_t *q_idx_scale, const float *head_w,
                            const void *k_idx_cache, const uint8_t *k_idx_scale, int64_t num_pages,
                            const int32_t *page_table, int32_t max_pages_per_seq, const int32_t *seq_lens,
                            const int32_t *cu_q, int32_t B, int32_t T, int32_t K, int32_t page_size,
                            dsa_idx_dtype dtype, int32_t *indices, float *scores, int64_t ld_scores,
                            void *workspace, size_t workspace_bytes, void *stream) {
    if (!scores || ld_scores < 1) return DSA_ERR_INVALID_ARG;
    return index_common(q_idx, q_idx_scale, head_w, k_idx_cache, k_idx_scale, num_pages, page_table,
                        max_pages_per_seq, seq_lens, cu_q, B, T, K, page_size, dtype, indices, scores, ld_scores,
                        workspace, workspace_bytes, stream);
}

dsa_status dsa_topk_from_scores(const float *scores, int64_t ld, const int32_t *lens, int32_t R, int32_t K,
                                int32_t *out, void *workspace, size_t workspace_bytes, void *stream) {
    if (!scores || !lens || !out || !workspace || R < 0 || K < 1 || ld < 1 || workspace_bytes < kErrBytes)
        return DSA_ERR_INVALID_ARG;
    if (R == 0) return DSA_OK;
    if (ld > (1LL << 30) || R > 65535) return DSA_ERR_UNSUPPORTED;
    const size_t smax = max_smem_optin();
    int forced = g_topk_cluster.load();
    for (int C = 1; C <= 16; C <<= 1) {
        if (forced && C != forced) continue;
        const int cap = ceil_div(ld, C);
        if (!forced && C < 16 && cap > 8192) continue;
        const size_t smem = dsa::topk_smem_bytes(cap);
        if (smem > smax) continue;
        TopkArgs a{scores, lens, out, ld, R, K, cap};
        return cuda_status(dsa::launch_topk_from_scores(a, C, smem, static_cast<cudaStream_t>(stream)));
    }
    return DSA_ERR_UNSUPPORTED;
}

dsa_status dsa_sparse_mla(const void *q, const void *kv_cache, const void *kv_rope, const float *kv_scale,
                          int64_t num_pages, const int32_t *page_table, int32_t max_pages_per_seq,
                          const int32_t *seq_lens, const int32_t *cu_q, const int32_t *indices, int32_t B,
                          int32_t T, int32_t H, int32_t K, float scale, int32_t page_size, dsa_kv_dtype dtype,
                          void *out, float *lse, void *workspace, size_t workspace_bytes, void *stream) {
    if (T < 0 || B < 1 || K < 1 || H < 1 || page_size < 1 || num_pages < 1 || max_pages_per_seq < 1)
        return DSA_ERR_INVALID_ARG;
    if (!q || !kv_cache || !page_table || !seq_lens || !cu_q || !indices || !out || !workspace)
        return DSA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(out) || !aligned16(workspace))
        return DSA_ERR_INVALID_ARG;
    const int NH = mla_heads_per_cta(H);
    if (NH == 0 || H > 1024 || T > 65535) return DSA_ERR_UNSUPPORTED;
    if ((long long)num_pages * page_size > (1LL << 31)) return DSA_ERR_UNSUPPORTED;
    if (dtype != DSA_KV_BF16 && dtype != DSA_KV_FP8_ROWSCALE && dtype != DSA_KV_FP8_TILE128)
        return DSA_ERR_UNSUPPORTED;
    const bool fp8 = dtype != DSA_KV_BF16;
    if (fp8 && (!kv_rope || !kv_scale || !aligned16(kv_rope) || (reinterpret_cast<uintptr_t>(kv_scale) & 3u)))
        return DSA_ERR_INVALID_ARG;
    // (a workspace of the split grid's size is enough: stream-K then stays off)
    if (workspace_bytes < split_workspace_size(T, H, K)) return DSA_ERR_INVALID_ARG;
    if (T == 0) return DSA_OK;
    const int splits = mla_splits(T, H, K);
    const int tile = dsa::mla_key_tile();
    MlaArgs a{};
    a.q = static_cast<const uint16_t *>(q);
    a.kv = static_cast<const uint8_t *>(kv_cache);
    a.kv_rope = fp8 ? static_cast<const uint8_t *>(kv_rope) : nullptr;
    a.kv_scale = fp8 ? kv_scale : nullptr;
    a.kv_scales = dtype == DSA_KV_FP8_TILE128 ? 4 : 1;
    a.page_table = page_table;
    a.seq_lens = seq_lens;
    a.cu_q = cu_q;
    a.indices = indices;
    a.out = static_cast<uint16_t *>(out);
    a.lse = lse;
    a.err = reinterpret_cast<uint32_t *>(workspace);
    const size_t rows = (size_t)T * mla_groups(H) * splits * 64;
    a.part_o = splits > 1 ? reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + kErrBytes) : nullptr;
    a.part_ml = splits > 1 ? a.part_o + rows * 512 : nullptr;
    a.num_pages = num_pages;
    a.max_pages = max_pages_per_seq;
    a.B = B;
    a.T = T;
    a.H = H;
    a.K = K;
    a.page_size = page_size;
    a.splits = splits;
    a.keys_per_split = ceil_div(ceil_div(K, splits), tile) * tile;
    a.scale = scale;
    a.scale_log2 = scale * 1.4426950408889634f;
    if (mla_dsplit(T, H, fp8, splits))
        return cuda_status(dsa::launch_sparse_mla_ds(a, static_cast<cudaStream_t>(stream)));
    const bool pair = mla_pair(T, H, splits);
    const int sk = pair ? 0 : mla_sk_ctas(T, H, K);
    if (sk > 0 && workspace_bytes >= mla_sk_workspace(sk)) {
        a.sk_ctas = sk;
        a.sk_tpr = ceil_div(K, tile);
        a.sk_units = (int64_t)T * a.sk_tpr;
        a.part_o = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + kErrBytes);
        a.part_ml = a.part_o + (size_t)2 * sk * 64 * 512;
    }
    CUtensorMap tq;
    if (!encode_2d_bf16(&tq, q, 576, (uint64_t)T * H, (uint32_t)NH)) return DSA_ERR_CUDA;
    return cuda_status(
        dsa::launch_sparse_mla(tq, a, NH, fp8, pair, static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_quant_mxfp8(const void *x, int64_t n, void *q, void *e8m0, void *stream) {
    if (n < 0 || n % 32 != 0 || (n > 0 && (!x || !q || !e8m0))) return DSA_ERR_INVALID_ARG;
    if (n > 0 && (!aligned16(x) || !aligned16(q))) return DSA_ERR_INVALID_ARG;
    return cuda_status(dsa::launch_quant_mxfp8(static_cast<const uint16_t *>(x), n, static_cast<uint8_t *>(q),
                                               static_cast<uint8_t *>(e8m0), static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_quant_fp8_rows(const void *kv, int64_t rows, void *nope, void *rope, float *scale, void *stream) {
    if (rows < 0 || (rows > 0 && (!kv || !nope || !rope || !scale))) return DSA_ERR_INVALID_ARG;
    if (rows > 0 && (!aligned16(kv) || !aligned16(nope) || (reinterpret_cast<uintptr_t>(rope) & 3u)))
        return DSA_ERR_INVALID_ARG;
    return cuda_status(dsa::launch_quant_fp8_rows(static_cast<const uint16_t *>(kv), rows,
                                                  static_cast<uint8_t *>(nope), static_cast<uint16_t *>(rope), scale,
                                                  static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_cache_append(const void *k_new, const void *kv_new, const int32_t *page_table,
                            int32_t max_pages_per_seq, const int32_t *seq_lens, const int32_t *cu_q, int32_t B,
                            int32_t T, int32_t page_size, int64_t num_pages, dsa_idx_dtype idx_dtype, void *k_cache,
                            void *k_scale, dsa_kv_dtype kv_dtype, void *kv_cache, void *kv_rope, float *kv_scale,
                            void *workspace, size_t workspace_bytes, void *stream) {
    const bool do_k = k_new != nullptr && k_cache != nullptr, do_kv = kv_new != nullptr && kv_cache != nullptr;
    if (T < 0 || B < 0 || (T > 0 && B == 0) || page_size <= 0 || num_pages < 0 || max_pages_per_seq < 0)
        return DSA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < kErrBytes || !aligned16(workspace)) return DSA_ERR_INVALID_ARG;
    if (idx_dtype != DSA_IDX_BF16 && idx_dtype != DSA_IDX_MXFP8) return DSA_ERR_UNSUPPORTED;
    if (kv_dtype != DSA_KV_BF16 && kv_dtype != DSA_KV_FP8_ROWSCALE && kv_dtype != DSA_KV_FP8_TILE128)
        return DSA_ERR_UNSUPPORTED;
    if (T == 0 || (!do_k && !do_kv)) return DSA_OK;
    if (!page_table || !seq_lens || !cu_q) return DSA_ERR_INVALID_ARG;
    if (do_k && (!aligned16(k_new) || !aligned16(k_cache) || (idx_dtype == DSA_IDX_MXFP8 && !k_scale)))
        return DSA_ERR_INVALID_ARG;
    const bool kv_fp8 = kv_dtype != DSA_KV_BF16;
    if (do_kv && (!aligned16(kv_new) || !aligned16(kv_cache) ||
                  (kv_fp8 && (!kv_rope || !kv_scale || (reinterpret_cast<uintptr_t>(kv_rope) & 3u) ||
                              (reinterpret_cast<uintptr_t>(kv_scale) & 3u)))))
        return DSA_ERR_INVALID_ARG;
    AppendArgs a{};
    a.k_new = do_k ? static_cast<const uint16_t *>(k_new) : nullptr;
    a.kv_new = do_kv ? static_cast<const uint16_t *>(kv_new) : nullptr;
    a.page_table = page_table;
    a.seq_lens = seq_lens;
    a.cu_q = cu_q;
    a.max_pages = max_pages_per_seq;
    a.B = B;
    a.page_size = page_size;
    a.T = T;
    a.num_pages = num_pages;
    a.k_cache = do_k ? k_cache : nullptr;
    a.k_scale = static_cast<uint8_t *>(k_scale);
    a.kv_cache = do_kv ? kv_cache : nullptr;
    a.kv_rope = static_cast<uint16_t *>(kv_rope);
    a.kv_scale = kv_scale;
    a.err = reinterpret_cast<uint32_t *>(workspace);
    const int kv_scales = kv_dtype == DSA_KV_BF16 ? 0 : (kv_dtype == DSA_KV_FP8_TILE128 ? 4 : 1);
    return cuda_status(dsa::launch_cache_append(a, idx_dtype == DSA_IDX_MXFP8, kv_scales,
                                                static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_quant_fp8_tiles(const void *kv, int64_t rows, void *nope, void *rope, float *scale, void *stream) {
    if (rows < 0 || (rows > 0 && (!kv || !nope || !rope || !scale))) return DSA_ERR_INVALID_ARG;
    if (rows > 0 && (!aligned16(kv) || !aligned16(nope) || (reinterpret_cast<uintptr_t>(rope) & 3u) ||
                     (reinterpret_cast<uintptr_t>(scale) & 3u)))
        return DSA_ERR_INVALID_ARG;
    return cuda_status(dsa::launch_quant_fp8_tiles(static_cast<const uint16_t *>(kv), rows,
                                                   static_cast<uint8_t *>(nope), static_cast<uint16_t *>(rope), scale,
                                                   static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
