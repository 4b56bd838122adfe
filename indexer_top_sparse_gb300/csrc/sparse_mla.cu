// sparse_mla.cu -- sparse MLA attention over the indexer's selected rows.
//
// What it computes ("Day0 Inference Support and Performance Optimization for
// New-Architecture LLMs", §2 item 2 and §4 "Sparse attention reads by index";
// "Day0 Inference Optimization for a New Hybrid Attention Architecture: A
// Full-Stack Deep Dive", operator fusion item 1): for query row t and head h,
//     out[t][h] = sum_i softmax_i(scale * q[t][h] . kv[idx_i]) * kv[idx_i][0:512]
// over the valid selected positions idx_i of row t only; the other cache rows
// are never read.
//
// Design (tcgen05, accumulators in TMEM).  CTA = (group of NH <= 64 heads,
// key split, query row); selected keys are processed in tiles of 64, two
// tiles in flight (a ring of shared-memory buffers).  With 128 heads the two
// 64-head CTAs of a query row form a cluster: each gathers half of every tile
// and forwards it to the other over distributed shared memory, so that every
// selected row is read from memory once.
//   warps 0-7   gather: every selected key of the split is first resolved to
//               its physical cache row (one table, built up front); then
//               16-byte cp.async copies place each 576-wide bf16 row into nine
//               64-column regions in the 128-byte-swizzle layout.  For the FP8
//               cache the 512 E4M3 latent dims go through registers (loaded a
//               tile ahead), are multiplied by their scale (the row's, or
//               the one of their 128-dim tile) and stored as
//               bf16; the rope dims are copied as they are.
//   warps 8, 13 tcgen05 issuers (split grid: even and odd tiles; stream-K:
//               warp 8 alone): S[64 heads x 64 keys] = Q . K_tile^T (M = 64,
//               K-major operands, 36 steps of K = 16, double-buffered in
//               TMEM; with a bf16 cache the first 12 steps start once regions
//               0-2 have landed), then O^T[512 dims x 64] += V^T . P^T with V^T
//               read MN-major from the same tile and P^T MN-major (4 chunks of
//               128 dims, 4 steps of 16 keys).
//               With pairs, each gather warp forwards its rows to the peer
//               (bulk shared-to-shared copies) as soon as they have landed.
//   warps 9-12  softmax: thread = head (M = 64 places rows 16q..16q+15 in the
//               low 16 lanes of warp quadrant q), so max, exp2 and sum over
//               the tile's keys stay in registers; the reference max moves
//               only when a head's max grows by more than 2^8, and then the
//               O^T columns are rescaled in TMEM; P (bf16) is written over the
//               tile's consumed rope region as [key][head] rows.  The same
//               warps run the epilogue.
// With several key splits per row, partial (O, max, sum) go to the workspace
// and mla_combine_kernel merges them.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math_constants.h>

#include "ptx.cuh"
#include "kernels.h"

namespace dsa {

namespace {

constexpr int kD = 576;
constexpr int kDv = 512;
constexpr int kHG = 64;                      // head-slot stride of the partial layout
constexpr int kKeys = 64;                    // keys per tile (MMA N of S; P rows are 128 bytes)
constexpr int kStages = 2;                   // tiles in flight
constexpr int kRegions = 9;                  // 64-dim regions of a 576-wide row
constexpr int kRegionBytes = kKeys * 128;    // 4 or 8 KB
constexpr int kTileBytes = kRegions * kRegionBytes;
constexpr int kQRegion = 64 * 128;           // Q rows padded to the MMA's M = 64
#ifndef MLA_PRODUCER_WARPS
#define MLA_PRODUCER_WARPS 8
#endif
constexpr int kProd = MLA_PRODUCER_WARPS;
constexpr int kMmaWarp = kProd;
constexpr int kSmWarp0 = kProd + 1;          // 4 softmax / epilogue warps
// Second tcgen05 issuer (split mode): kMmaWarp issues the logits and P*V of
// the even tiles, kMmaWarp2 those of the odd tiles, so that the logits of the
// next tile are issued while this tile's softmax runs (one thread's issues
// and waits for a tile take longer than the tensor core needs for them).
constexpr int kMmaWarp2 = kSmWarp0 + 4;
constexpr int kThreads = (kProd + 1 + 4 + 1) * 32;
constexpr int kSmThreads = 128;
constexpr int kBarSm = 1;
constexpr int kBarProd = 2;
static_assert(kKeys % kProd == 0, "gather work splits evenly");
constexpr int kWords = kKeys / 32;           // validity words per tile

template <int NH>
struct MlaLayout {
    static constexpr int kKVOff = kRegions * kQRegion;
    static constexpr int kMiscOff = kKVOff + kStages * kTileBytes;
    static constexpr int kTmemCols = 512;    // O^T: 4 chunks x 64 columns at 0; S buffers at 256 + 32 j
};

struct __align__(16) MlaBars {
    uint64_t kv_full[kStages], kv_empty[kStages], s_full[2];
    // bf16 cache, unpaired: the first kEarlyRegions regions of the stage's
    // tile have landed (the logits start on them while the rest lands)
    uint64_t kv_early[kStages];
    uint64_t peer_free[kStages];   // pairs: the peer's copy of this stage may be overwritten
    // pairs: every byte of this CTA's half of the stage's tile has landed in
    // the peer, so the forwarding copies have finished reading it here and
    // the rope region may take P
    uint64_t fwd_done[kStages];
    uint64_t p_full[2];  // P of tile i is in its stage: p_full[i & 1]
    uint64_t drain[2];   // one per issuing thread
    uint64_t o_done, o_full, q_full, table;
    uint64_t o_free;  // stream-K: the epilogue of segment 0 has read O
    uint32_t tmem_slot;
    int abort[2];  // [0] a wait gave up; [1] wait limit in microseconds (0: default)
};

constexpr int kMaxKeysPerSplit = 2048;       // host keeps keys_per_split <= this
constexpr int kEarlyRegions = 3;             // regions behind kv_early (bf16 cache, unpaired)

struct __align__(16) MlaStats {
    int32_t rows[kMaxKeysPerSplit];             // physical cache row of every key of the split
    uint32_t valid[kMaxKeysPerSplit / 32];      // bit k%32 of word k/32: key k is valid
    float alpha[2][kHG];
    float m_fin[kHG];
    float l_fin[kHG];
};

__device__ __forceinline__ int find_seq(const int32_t *cu_q, int B, int t) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (__ldg(cu_q + mid) <= t) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ bool bar_or(int id, int count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %1, 0;\n\t"
        "barrier.cta.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// 16 E4M3 latent values (one lane's 16 bytes of a row) times the row scale,
// as 8 words of bf16 pairs (low half = lower dim).  E4M3 -> f16 -> f32 is
// exact; the product is rounded once, to bf16.
__device__ __forceinline__ void dequant16(const uint4 v, const float s, uint32_t out[8]) {
    const uint32_t in[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(in[i] >> (16 * h)), __NV_E4M3);
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&r));
            out[2 * i + h] = pack_bf16(f.x * s, f.y * s);
        }
    }
}

// Issue S = Q . K_tile^T for tile i into S buffer i&1 once the tile landed
// (kEarly: the first kEarlyRegions regions' steps once those have landed,
// the rest once the whole tile has).
template <bool kEarly>
__device__ __forceinline__ bool issue_s_tile(int i, MlaBars *bars, uint32_t kv_base, uint32_t q_base, uint32_t tmem_s,
                                             uint32_t idesc_s, uint32_t *err, volatile int *abort, int wl) {
    const int st = i % kStages;
    // descriptors advance by (byte offset >> 4) in their start-address field
    const uint64_t ad0 = sdesc_kmajor_sw128(q_base);
    const uint64_t bd0 = sdesc_kmajor_sw128(kv_base + st * kTileBytes);
    const uint32_t d = tmem_s + kKeys * (i & 1);
#pragma unroll
    for (int r = 0; r < kRegions; ++r) {
        if (r == (kEarly ? kEarlyRegions : 0)) {
            if (!mbar_wait(&bars->kv_full[st], (i / kStages) & 1, err, 0x503, abort, wl)) return false;
            fence_proxy_async_smem();  // the tile was written through the generic proxy
            tc_fence_after();
        } else if (kEarly && r == 0) {
            if (!mbar_wait(&bars->kv_early[st], (i / kStages) & 1, err, 0x515, abort, wl)) return false;
            fence_proxy_async_smem();
            tc_fence_after();
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ss(d, ad0 + (uint64_t)((r * kQRegion + kk * 32) >> 4),
                        bd0 + (uint64_t)((r * kRegionBytes + kk * 32) >> 4), idesc_s, (r | kk) ? 1u : 0u);
    }
    mma_commit(&bars->s_full[i & 1]);
    return true;
}

// kPair: the two 64-head CTAs of a query row form a cluster; each gathers half
// of every tile (from global memory) and forwards it to the other's shared
// memory, so that each selected row is read from L2/HBM once.
// kF8: the cache holds E4M3 latent dims + an fp32 scale per row + bf16 rope
// dims; the gather warps dequantise the latent dims to bf16 through registers.
template <int NH, bool kPair, bool kF8, bool kSK>
__global__ void __launch_bounds__(kThreads, 1) sparse_mla_tc_kernel(const __grid_constant__ CUtensorMap tm_q, MlaArgs a) {
    using L = MlaLayout<NH>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQ = smem;
    uint8_t *sKV = smem + L::kKVOff;  // two tiles
    MlaBars *bars = reinterpret_cast<MlaBars *>(smem + L::kMiscOff);
    MlaStats *st = reinterpret_cast<MlaStats *>(bars + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // What this CTA computes: one or two segments, each a run of consecutive
    // key tiles of one (query row t, head group hg); tile i of the CTA
    // belongs to segment 1 from seg[1].first on.  Split mode: the grid is
    // (head group, key split, row), one segment.  Stream-K mode: one row of
    // CTAs shares all (row, head group, key tile) units evenly, and a CTA's
    // run may cross into the next (row, head group) once.
    struct Seg {
        int t, hg, j0, first;  // row, head group, its first key tile, first CTA-local tile
    };
    Seg seg[2];
    int n_seg = 1, n_tiles;
    if constexpr (kSK) {
        // each head group has sk_ctas / G CTAs that share its U = T * tpr
        // (row, key tile) units the same way, so the CTAs of the head groups
        // of a row gather the same rows at the same time
        const int G = a.H / NH;
        const int64_t Cg = a.sk_ctas / G, U = a.sk_units, c = blockIdx.x % Cg;
        const int tpr = a.sk_tpr;
        const int64_t u0 = c * U / Cg, u1 = (c + 1) * U / Cg;
        n_tiles = (int)(u1 - u0);
        const int64_t r0 = u0 / tpr, e0 = (r0 + 1) * tpr;
        seg[0] = {(int)r0, (int)(blockIdx.x / Cg), (int)(u0 - r0 * tpr), 0};
        seg[1] = seg[0];
        if (u1 > e0) {
            n_seg = 2;
            seg[1].t = (int)(r0 + 1);
            seg[1].j0 = 0;
            seg[1].first = (int)(e0 - u0);
        }
    } else {
        const int k_begin = blockIdx.y * a.keys_per_split;
        const int k_end = min(a.K, k_begin + a.keys_per_split);
        n_tiles = k_end > k_begin ? (k_end - k_begin + kKeys - 1) / kKeys : 0;
        seg[0] = {(int)blockIdx.z, (int)blockIdx.x, k_begin / kKeys, 0};
        seg[1] = seg[0];
    }
    const int s1 = n_seg == 2 ? seg[1].first : n_tiles;  // first tile of segment 1 (n_tiles if none)
    const int t = seg[0].t, hg = seg[0].hg;
    // segment of CTA-local tile i (always 0 in split mode); the per-segment
    // values are picked with selects, so that they stay in registers
    auto seg_of = [&](int i) { return kSK && i >= s1 ? 1 : 0; };
    // Inputs may come from the kernel launched just before this one (the
    // indexer's indices, or a caller's kernel); with programmatic dependent
    // launch this kernel starts early and waits here until they are visible.
    grid_dep_wait();
    auto seq_pos = [&](int tt, int &bb, int &pp) {
        bb = find_seq(a.cu_q, a.B, tt);
        pp = __ldg(a.seq_lens + bb) - (__ldg(a.cu_q + bb + 1) - __ldg(a.cu_q + bb)) + (tt - __ldg(a.cu_q + bb));
    };
    int sb0, spos0, sb1, spos1;
    seq_pos(seg[0].t, sb0, spos0);
    sb1 = sb0;
    spos1 = spos0;
    if (kSK && n_seg == 2) seq_pos(seg[1].t, sb1, spos1);

    if (threadIdx.x == 0) {
        // a tile is complete after one cp.async completion arrival per gather
        // lane, (FP8) one arrival per gather warp after its dequantised
        // stores, and (pairs) one arrival that expects the peer's half in bytes
        constexpr int kFullArrivals = 32 * kProd + (kF8 ? kProd : 0) + (kPair ? 1 : 0);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&bars->kv_full[i], kFullArrivals);
            mbar_init(&bars->kv_early[i], 32 * kProd);
            mbar_init(&bars->kv_empty[i], 1);
            mbar_init(&bars->peer_free[i], 1);
            mbar_init(&bars->fwd_done[i], 1);
        }
        for (int i = 0; i < 2; ++i) mbar_init(&bars->s_full[i], 1);
        mbar_init(&bars->p_full[0], kSmThreads / 32);
        mbar_init(&bars->p_full[1], kSmThreads / 32);
        mbar_init(&bars->o_done, 1);
        mbar_init(&bars->o_full, 1);
        mbar_init(&bars->o_free, kSmThreads / 32);
        mbar_init(&bars->q_full, 1);
        mbar_init(&bars->drain[0], 1);
        mbar_init(&bars->drain[1], 1);
        mbar_init(&bars->table, 1);
        bars->abort[0] = 0;
        bars->abort[1] = wait_limit_us(a.err);
        fence_mbar_init();
    }
    if constexpr (NH < 64) {
        // Q rows NH..63 feed MMA rows nobody reads; keep them finite
        for (int i = threadIdx.x; i < kRegions * (64 - NH) * 8; i += kThreads) {
            const int r = i / ((64 - NH) * 8), rem = i % ((64 - NH) * 8);
            reinterpret_cast<uint4 *>(sQ + r * kQRegion + NH * 128)[rem] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    if (warp == kMmaWarp) tmem_alloc(&bars->tmem_slot, L::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if constexpr (kPair) cluster_barrier();  // both CTAs' barriers are initialised before any remote arrive
    const uint32_t peer = kPair ? (cluster_rank() ^ 1u) : 0u;
    const uint32_t tmem_o = bars->tmem_slot;      // O^T chunk c: columns [64 c, 64 c + NH)
    const uint32_t tmem_s = tmem_o + 256;         // S buffer j at columns 256 + kKeys j (<= 384)
    volatile int *abort = bars->abort;
    const int wl = abort[1];  // test wait limit in microseconds (0: the default limit)

    if (warp < kProd) {
        // ---------------------------------------------------------------- gather
        // keys of a tile this CTA gathers: all of them, or its half when paired
        constexpr int kMine = kPair ? kKeys / 2 : kKeys;
        constexpr int kKPW = kMine / kProd;  // keys per gather warp
        static_assert(kKPW * 8 % 32 == 0 && kKPW <= 32, "a warp instruction covers four keys");
        const int key0 = (kPair ? (int)cluster_rank() * kMine : 0) + warp * kKPW;
        if (warp == 0 && lane == 0) {
            tma_prefetch_desc(&tm_q);
            mbar_arrive_expect_tx(&bars->q_full, (uint32_t)(kRegions * NH * 128));
            for (int r = 0; r < kRegions; ++r)
                tma_load_2d(sQ + r * kQRegion, &tm_q, &bars->q_full, 64 * r, t * a.H + hg * NH);
        }
        // resolve every selected key of the split to its physical row once,
        // in parallel, so that the copy loop below never waits on the index
        // or page-table loads
        const int n_keys = n_tiles * kKeys;
        constexpr int kPer = kMaxKeysPerSplit / (kProd * 32);  // keys per gather thread, at most
        int idxv[kPer], pagev[kPer];
        // all index loads first, then all page-table loads, then the table
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int k = threadIdx.x + u * kProd * 32, i = k / kKeys, s = seg_of(i);
            const int j0 = s ? seg[1].j0 : seg[0].j0, first = s ? seg[1].first : 0, tt = s ? seg[1].t : seg[0].t;
            const int slot = (j0 + i - first) * kKeys + k % kKeys;
            idxv[u] = k < n_keys && slot < a.K ? __ldg(a.indices + (size_t)tt * a.K + slot) : -1;
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int k = threadIdx.x + u * kProd * 32, s = seg_of(k / kKeys);
            const int pos = s ? spos1 : spos0, bb = s ? sb1 : sb0;
            // a position past the sequence's page-table row (seq_lens larger
            // than max_pages * page_size) is reported as a bad page, unread
            pagev[u] = idxv[u] >= 0 && idxv[u] <= pos && idxv[u] / a.page_size < a.max_pages
                           ? __ldg(a.page_table + (size_t)bb * a.max_pages + idxv[u] / a.page_size)
                           : -1;
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int k = threadIdx.x + u * kProd * 32;
            if (k >= n_keys) break;  // n_keys is a multiple of 64: warp-uniform
            const int idx = idxv[u], pos = seg_of(k / kKeys) ? spos1 : spos0;
            int row = 0;  // invalid slots read row 0 and are masked by the softmax
            bool v = false;
            if (idx > pos) {
                report_error(a.err, kErrBadIndex);
            } else if (idx >= 0) {
                const int page = pagev[u];
                if (page < 0 || (int64_t)page >= a.num_pages) {
                    report_error(a.err, kErrBadPage);
                } else {
                    row = page * a.page_size + idx % a.page_size;
                    v = true;
                }
            }
            st->rows[k] = row;
            const uint32_t bits = __ballot_sync(0xffffffffu, v);
            if (lane == 0) st->valid[k >> 5] = bits;
        }
        bar_sync(kBarProd, kProd * 32);  // gather warps only
        if (threadIdx.x == 0) mbar_arrive(&bars->table);  // publishes the row / validity table
        // FP8: lane l holds bytes 16l..16l+15 (dims 16l..16l+15) of each of
        // the warp's keys, loaded one tile ahead so that the loads overlap the
        // wait for a free stage
        uint4 f8v[kF8 ? kKPW : 1];
        float f8s[kF8 ? kKPW : 1];
        if constexpr (kF8) {
            if (n_tiles > 0) {
#pragma unroll
                for (int j = 0; j < kKPW; ++j) {
                    const int row = st->rows[key0 + j];
                    f8v[j] = __ldg(reinterpret_cast<const uint4 *>(a.kv + (size_t)row * kDv) + lane);
                    f8s[j] = __ldg(a.kv_scale + (size_t)row * a.kv_scales + ((lane * a.kv_scales) >> 5));
                }
            }
        }
        for (int i = 0; i < n_tiles; ++i) {
            const int stg = i % kStages;
            bool ok = true;
            if (i >= kStages) ok = mbar_wait(&bars->kv_empty[stg], ((i / kStages) & 1) ^ 1, a.err, 0x501, abort, wl);
            if (!__all_sync(0xffffffffu, ok)) break;
            if (kPair && threadIdx.x == 0) {
                // this stage is free here: the peer may send its half of tile i
                mbar_arrive_remote(map_peer(smem_u32(&bars->peer_free[stg]), peer));
                mbar_arrive_expect_tx(&bars->kv_full[stg], kRegions * kMine * 128);
            }
            uint8_t *dst = sKV + stg * kTileBytes;
            const int32_t *rows = st->rows + i * kKeys;
            uint64_t *done = &bars->kv_full[stg];
            if constexpr (!kF8) {
                // (unpaired: the first kEarlyRegions regions complete kv_early)
                auto copy_regions = [&](int r0, int r1) {
#pragma unroll 3
                    for (int r = r0; r < r1; ++r) {
#pragma unroll
                        for (int m = 0; m < kKPW * 8 / 32; ++m) {
                            const int f = m * 32 + lane, key = key0 + (f >> 3), cc = f & 7;
                            const uint8_t *src = a.kv + (size_t)rows[key] * (kD * 2) + r * 128 + cc * 16;
                            cp_async16(dst + r * kRegionBytes + key * 128 + ((cc ^ (key & 7)) << 4), src);
                        }
                    }
                };
                if constexpr (!kPair) {
                    copy_regions(0, kEarlyRegions);
                    cp_async_arrive(&bars->kv_early[stg]);
                    copy_regions(kEarlyRegions, kRegions);
                } else {
                    copy_regions(0, kRegions);
                }
                cp_async_arrive(done);
            } else {
                // rope dims (bf16) straight into region 8
#pragma unroll
                for (int m = 0; m < kKPW * 8 / 32; ++m) {
                    const int f = m * 32 + lane, key = key0 + (f >> 3), cc = f & 7;
                    cp_async16(dst + 8 * kRegionBytes + key * 128 + ((cc ^ (key & 7)) << 4),
                               a.kv_rope + (size_t)rows[key] * 128 + cc * 16);
                }
                cp_async_arrive(done);
                // latent dims: lane l fills 16-byte chunks 2(l%4), 2(l%4)+1 of
                // region l/4; odd regions store the odd chunk first, so each
                // store instruction covers all eight chunk positions (banks)
                const int r = lane >> 2, c0 = (lane & 3) * 2, flip = r & 1;
#pragma unroll
                for (int j = 0; j < kKPW; ++j) {
                    const int key = key0 + j;
                    uint32_t w[8];
                    dequant16(f8v[j], f8s[j], w);
                    uint8_t *base = dst + r * kRegionBytes + key * 128;
                    const uint4 lo = make_uint4(w[0], w[1], w[2], w[3]), hi = make_uint4(w[4], w[5], w[6], w[7]);
                    *reinterpret_cast<uint4 *>(base + (((c0 + flip) ^ (key & 7)) << 4)) = flip ? hi : lo;
                    *reinterpret_cast<uint4 *>(base + (((c0 + 1 - flip) ^ (key & 7)) << 4)) = flip ? lo : hi;
                }
                fence_proxy_async_smem();  // the tensor cores (or the pair copy) read these stores
                __syncwarp();
                if (lane == 0) mbar_arrive(done);
                if (i + 1 < n_tiles) {
                    const int32_t *nrows = rows + kKeys;
#pragma unroll
                    for (int j = 0; j < kKPW; ++j) {
                        const int row = nrows[key0 + j];
                        f8v[j] = __ldg(reinterpret_cast<const uint4 *>(a.kv + (size_t)row * kDv) + lane);
                        f8s[j] = __ldg(a.kv_scale + (size_t)row * a.kv_scales + ((lane * a.kv_scales) >> 5));
                    }
                }
            }
            if constexpr (kPair) {
                // forward this warp's keys (kKPW rows of every region) to the
                // peer as soon as they have landed here
                cp_async_wait_all();
                fence_proxy_async_smem();  // written through the generic proxy, read by the bulk copy
                __syncwarp();
                if (lane == 0) {
                    ok = mbar_wait(&bars->peer_free[stg], (i / kStages) & 1, a.err, 0x512, abort, wl);
                    if (ok) {
                        const uint32_t rbar = map_peer(smem_u32(&bars->kv_full[stg]), peer);
                        for (int r = 0; r < kRegions; ++r) {
                            uint8_t *src = dst + r * kRegionBytes + key0 * 128;
                            bulk_copy_to_peer(map_peer(smem_u32(src), peer), src, kKPW * 128, rbar);
                        }
                    }
                }
                if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            }
        }
        cp_async_wait_all();  // the CTA stays alive until every copy has landed
        if (warp == 0 && lane == 0 && *abort) {
            volatile int no_abort[2] = {0, 0};
            mbar_wait(&bars->q_full, 0, nullptr, 0, no_abort);
        }
    } else if (warp == kMmaWarp || warp == kMmaWarp2) {
        // ---------------------------------------------------------------- tcgen05 issuers
        constexpr uint32_t idesc_s = idesc_bf16_f32(64, kKeys);
        // P*V always runs with N = 64 (all 64 rows of P); columns NH..63
        // are unused when NH < 64
        constexpr uint32_t idesc_o = idesc_bf16_f32_amn(128, 64);  // A (V^T) MN-major, B (P) K-major
        const uint32_t q_base = smem_u32(sQ), kv_base = smem_u32(sKV);
        uint32_t *const err = a.err;
        if (!kSK && lane == 0) {
            // split mode: tile i's logits and P*V by kMmaWarp (i even) or
            // kMmaWarp2 (i odd).  Logits of tile i go to S buffer i & 1, which
            // the softmax of tile i - 2 has read (p_full) before this thread
            // issued that tile's P*V; P*V of tile i follows the softmax of tile
            // i, which waited for P*V of tile i - 1 (o_done), so the additions
            // into O^T stay in tile order.
            const int par = warp == kMmaWarp ? 0 : 1;
            bool ok = mbar_wait(&bars->q_full, 0, a.err, 0x502, abort, wl);
            for (int i = par; ok && i < n_tiles; i += 2) {
                if (!(ok = issue_s_tile<!kPair && !kF8>(i, bars, kv_base, q_base, tmem_s, idesc_s, err, abort, wl))) break;
                if (!(ok = mbar_wait(&bars->p_full[i & 1], (i >> 1) & 1, a.err, 0x504, abort, wl))) break;
                tc_fence_after();
                const int stg = i % kStages;
                const uint32_t kb = kv_base + stg * kTileBytes;
                const uint64_t ad0 = sdesc_mnmajor_sw128(kb, kRegionBytes, 1024);
                const uint64_t bd0 = sdesc_kmajor_sw128(kb + 8 * kRegionBytes);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
#pragma unroll
                    for (int j = 0; j < kKeys / 16; ++j)
                        mma_bf16_ss(tmem_o + c * 64, ad0 + (uint64_t)((2 * c * kRegionBytes + j * 2048) >> 4),
                                    bd0 + (uint64_t)((j * 32) >> 4), idesc_o, (i > 0 || j > 0) ? 1u : 0u);
                }
                mma_commit(&bars->kv_empty[stg]);
                mma_commit(&bars->o_done);
                // every earlier P*V has completed (o_done of tile i - 1 came before P of tile i)
                if (i + 1 == n_tiles) mma_commit(&bars->o_full);
            }
            if (*abort) {
                volatile int no_abort[2] = {0, 0};
                mma_commit(&bars->drain[par]);
                mbar_wait(&bars->drain[par], 0, nullptr, 0, no_abort);
            }
        } else if (kSK && warp == kMmaWarp && lane == 0) {
            bool ok = mbar_wait(&bars->q_full, 0, a.err, 0x502, abort, wl);
            // Before the logits of segment 1's first tile: the last logits of
            // segment 0 have read Q, so its rows are replaced by segment 1's.
            auto switch_q = [&](int i) -> bool {
                if (!kSK || i != s1 || n_seg != 2) return true;
                if (!mbar_wait(&bars->s_full[(i - 1) & 1], ((i - 1) >> 1) & 1, a.err, 0x50a, abort, wl)) return false;
                mbar_arrive_expect_tx(&bars->q_full, (uint32_t)(kRegions * NH * 128));
                for (int r = 0; r < kRegions; ++r)
                    tma_load_2d(sQ + r * kQRegion, &tm_q, &bars->q_full, 64 * r, seg[1].t * a.H + seg[1].hg * NH);
                return mbar_wait(&bars->q_full, 1, a.err, 0x50b, abort, wl);
            };
            if (ok && n_tiles > 0) ok = issue_s_tile<!kPair && !kF8>(0, bars, kv_base, q_base, tmem_s, idesc_s, err, abort, wl);
            for (int i = 0; ok && i < n_tiles; ++i) {
                // With a ring of 3+ tiles the next tile's logits are issued
                // first, so that they overlap this tile's softmax; with only
                // 2 buffers the next tile is still loading, so this tile's
                // P*V goes first (it frees the buffer the tile after needs).
                if (kStages > 2 && i + 1 < n_tiles &&
                    !(ok = switch_q(i + 1) && issue_s_tile<!kPair && !kF8>(i + 1, bars, kv_base, q_base, tmem_s, idesc_s, err, abort, wl)))
                    break;
                if (!(ok = mbar_wait(&bars->p_full[i & 1], (i >> 1) & 1, a.err, 0x504, abort, wl))) break;
                // segment 1 starts a fresh accumulator once segment 0's epilogue has read O
                const int first = seg_of(i) ? s1 : 0;
                if (kSK && i == s1 && !(ok = mbar_wait(&bars->o_free, 0, a.err, 0x50c, abort, wl))) break;
                tc_fence_after();
                const int stg = i % kStages;
                const uint32_t kb = kv_base + stg * kTileBytes;
                // P [heads][keys] (K-major) over the consumed rope region
                const uint64_t ad0 = sdesc_mnmajor_sw128(kb, kRegionBytes, 1024);
                const uint64_t bd0 = sdesc_kmajor_sw128(kb + 8 * kRegionBytes);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
#pragma unroll
                    for (int j = 0; j < kKeys / 16; ++j)
                        mma_bf16_ss(tmem_o + c * 64, ad0 + (uint64_t)((2 * c * kRegionBytes + j * 2048) >> 4),
                                    bd0 + (uint64_t)((j * 32) >> 4), idesc_o, (i > first || j > 0) ? 1u : 0u);
                }
                mma_commit(&bars->kv_empty[stg]);
                mma_commit(&bars->o_done);
                if (i + 1 == s1 && s1 < n_tiles) mma_commit(&bars->o_full);  // segment 0 is complete
                if (kStages <= 2 && i + 1 < n_tiles &&
                    !(ok = switch_q(i + 1) && issue_s_tile<!kPair && !kF8>(i + 1, bars, kv_base, q_base, tmem_s, idesc_s, err, abort, wl)))
                    break;
            }
            if (ok && n_tiles > 0) mma_commit(&bars->o_full);
            if (*abort) {
                volatile int no_abort[2] = {0, 0};
                mma_commit(&bars->drain[0]);
                mbar_wait(&bars->drain[0], 0, nullptr, 0, no_abort);
            }
        } else if (kPair && warp == kMmaWarp && lane == 1) {
            // Pairs: tell the peer as soon as each tile -- including the half
            // the peer forwarded -- has landed here; the peer then knows that
            // its forwarding copies have read the rows it may overwrite.
            const uint32_t fwd_peer = map_peer(smem_u32(&bars->fwd_done[0]), peer);
            for (int i = 0; i < n_tiles; ++i) {
                const int stg = i % kStages;
                if (!mbar_wait(&bars->kv_full[stg], (i / kStages) & 1, a.err, 0x514, abort, wl)) break;
                mbar_arrive_remote(fwd_peer + 8 * stg);
            }
        }
    } else {
        // ---------------------------------------------------------------- softmax + epilogue
        const int sw = warp - kSmWarp0, quad = warp & 3;
        const int tid_s = sw * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        // With M = 64, S rows (heads) 16q..16q+15 sit in the first 16 lanes of
        // quadrant q; the 16x256b load spreads them over the whole warp:
        // thread = heads hA, hB (= hA + 8) x keys 8j + kc + {0, 1}.
        const int hA = quad * 16 + (lane >> 2), hB = hA + 8;
        const int kc = 2 * (lane & 3);
        const bool lead = (lane & 3) == 0;  // writes the per-head values
        float m_ref[2] = {-CUDART_INF_F, -CUDART_INF_F}, l_run[2] = {0.0f, 0.0f};
        bool ok = n_tiles == 0 || mbar_wait(&bars->table, 0, a.err, 0x509, abort, wl);
        // Epilogue of segment s: O / l (or the partial O, max and sum) for its
        // row and head group.  Segment 0 of a two-segment CTA runs inside the
        // tile loop and then hands O over to segment 1 (o_free).
        auto epilogue = [&](int s, bool last) {
            if (lead) {
                if (hA < NH) {
                    st->m_fin[hA] = m_ref[0];
                    st->l_fin[hA] = l_run[0];
                }
                if (hB < NH) {
                    st->m_fin[hB] = m_ref[1];
                    st->l_fin[hB] = l_run[1];
                }
            }
            if (last && tid_s == 0) grid_dep_launch();  // the split combine may start launching
            if (ok && n_tiles > 0) ok = mbar_wait(&bars->o_full, (uint32_t)s & 1u, a.err, 0x508, abort, wl);
            ok = bar_and(kBarSm, kSmThreads, ok);
            if (!ok) return;
            tc_fence_after();
            const int groups = a.H / NH, tt = s ? seg[1].t : seg[0].t, hgs = s ? seg[1].hg : seg[0].hg;
            const int h_base = hgs * NH;
            const bool direct = !kSK && a.splits == 1;
            // partial slot: stream-K (CTA, segment), else (row, head group, split)
            const size_t slot_base = kSK ? ((size_t)blockIdx.x * 2 + s) * kHG
                                         : (((size_t)tt * groups + hgs) * a.splits + blockIdx.y) * kHG;
            constexpr int W = NH < 32 ? NH : 32;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                const int d = c * 128 + quad * 32 + lane;
#pragma unroll
                for (int h0 = 0; h0 < NH; h0 += W) {
                    uint32_t o[W];
                    if (n_tiles > 0) {
                        tmem_ld<W>(tmem_o + lane_off + c * 64 + h0, o);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int j = 0; j < W; ++j) o[j] = 0u;
                    }
                    if (direct) {
#pragma unroll
                        for (int j = 0; j < W; ++j) {
                            const float l = st->l_fin[h0 + j];
                            const float v = l > 0.0f ? __uint_as_float(o[j]) / l : 0.0f;
                            a.out[((size_t)tt * a.H + h_base + h0 + j) * kDv + d] =
                                __bfloat16_as_ushort(__float2bfloat16_rn(v));
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < W; ++j) a.part_o[(slot_base + h0 + j) * kDv + d] = __uint_as_float(o[j]);
                    }
                }
            }
            if (tid_s < NH) {
                const float l = st->l_fin[tid_s], m = st->m_fin[tid_s];
                if (direct) {
                    if (a.lse)
                        a.lse[(size_t)tt * a.H + h_base + tid_s] =
                            l > 0.0f ? m * 0.69314718055994531f + logf(l) : -CUDART_INF_F;
                } else {
                    a.part_ml[(slot_base + tid_s) * 2 + 0] = l > 0.0f ? m : -CUDART_INF_F;
                    a.part_ml[(slot_base + tid_s) * 2 + 1] = l;
                }
            }
            if (!last) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->o_free);  // O may be overwritten
            }
        };
        for (int i = 0; i < n_tiles; ++i) {
            const int sb = i & 1, stg = i % kStages;
            if (kSK && i == s1) {
                // segment 0 is done: write it out, start segment 1 afresh
                epilogue(0, false);
                if (!ok) break;
                m_ref[0] = m_ref[1] = -CUDART_INF_F;
                l_run[0] = l_run[1] = 0.0f;
            }
            ok = mbar_wait(&bars->s_full[sb], (i >> 1) & 1, a.err, 0x505, abort, wl);
            ok = bar_and(kBarSm, kSmThreads, ok);
            if (!ok) break;
            tc_fence_after();
            constexpr int kJ = kKeys / 8;  // 8-column chunks
            float x[2][2 * kJ];
            {
                uint32_t r[4 * kJ];
                tmem_ld16x256b_x8(tmem_s + kKeys * sb + lane_off, r);
                tmem_wait_ld();
                const uint32_t v0 = st->valid[i * kWords], v1 = st->valid[i * kWords + 1];
#pragma unroll
                for (int j = 0; j < kJ; ++j) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int key = 8 * j + kc + e;
                        const bool valid = (((j < 4 ? v0 : v1) >> (key & 31)) & 1u) != 0;
                        x[0][2 * j + e] = valid ? __uint_as_float(r[4 * j + e]) * a.scale_log2 : -CUDART_INF_F;
                        x[1][2 * j + e] = valid ? __uint_as_float(r[4 * j + 2 + e]) * a.scale_log2 : -CUDART_INF_F;
                    }
                }
            }
            float al[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                float m4[4] = {x[u][0], x[u][1], x[u][2], x[u][3]};
#pragma unroll
                for (int k = 4; k < 2 * kJ; ++k) m4[k & 3] = fmaxf(m4[k & 3], x[u][k]);
                float mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
                al[u] = 1.0f;
                if (mt != -CUDART_INF_F && (m_ref[u] == -CUDART_INF_F || mt > m_ref[u] + 8.0f)) {
                    al[u] = m_ref[u] == -CUDART_INF_F ? 1.0f : exp2f(m_ref[u] - mt);
                    m_ref[u] = mt;
                }
                const float ref = m_ref[u] == -CUDART_INF_F ? 0.0f : m_ref[u];
                float s4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int k = 0; k < 2 * kJ; ++k) {
                    x[u][k] = exp2f(x[u][k] - ref);
                    s4[k & 3] += x[u][k];
                }
                float sum = (s4[0] + s4[1]) + (s4[2] + s4[3]);
                sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                l_run[u] = l_run[u] * al[u] + sum;
            }
            if (lead) {
                if (hA < NH) st->alpha[sb][hA] = al[0];
                if (hB < NH) st->alpha[sb][hB] = al[1];
            }
            // pairs: the rope rows this CTA forwarded from this stage must have
            // been read by their copies (they have landed in the peer) before
            // P overwrites them
            if (kPair && ok) ok = mbar_wait<true>(&bars->fwd_done[stg], (i / kStages) & 1, a.err, 0x513, abort, wl);
            {
                // P (bf16) as K-major [head][key] rows of 128 bytes with the
                // 128-byte swizzle, over the tile's consumed rope region (the
                // previous tile's P*V reads the other buffer)
                uint8_t *pb = sKV + stg * kTileBytes + 8 * kRegionBytes;
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int h = u ? hB : hA;
                    uint8_t *row = pb + h * 128 + 2 * kc;
#pragma unroll
                    for (int j = 0; j < kJ; ++j)
                        *reinterpret_cast<uint32_t *>(row + ((j ^ (h & 7)) << 4)) = pack_bf16(x[u][2 * j], x[u][2 * j + 1]);
                }
            }
            // O^T of the previous tile must be complete before it is rescaled
            if (i > 0) ok = mbar_wait(&bars->o_done, (i - 1) & 1, a.err, 0x507, abort, wl);
            const bool any = bar_or(kBarSm, kSmThreads,
                                    lead && ((hA < NH && al[0] != 1.0f) || (hB < NH && al[1] != 1.0f)));
            if (any && i > 0) {
                // rescale the O^T columns (heads) of this warp's 32 value-dim lanes
                // (a rare path: 16 columns at a time keeps registers free)
                constexpr int W = 16;
#pragma unroll 1
                for (int cc = 0; cc < 4 * (NH / W); ++cc) {
                    {
                        const int c = cc / (NH / W), h0 = (cc % (NH / W)) * W;
                        uint32_t o[W];
                        const uint32_t ta = tmem_o + lane_off + c * 64 + h0;
                        tmem_ld<W>(ta, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < W; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * st->alpha[sb][h0 + j]);
                        tmem_st<W>(ta, o);
                    }
                }
                tmem_wait_st();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->p_full[i & 1]);
        }
        // ---------------------------------------------------------------- epilogue
        epilogue(n_seg - 1, true);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem_o, L::kTmemCols);
    // no CTA of a pair leaves while the other may still signal or copy into it
    if constexpr (kPair) cluster_barrier();
}

// Merge split partials: block = (4 heads, head group, query row), warp = head,
// lane = 16 value dims (4 float4).  Splits are folded in with a running max, so
// every load of a split is independent of the previous split's arithmetic.
__global__ void __launch_bounds__(128) mla_combine_kernel(MlaArgs a, int NH) {
    const int hg = blockIdx.y, t = blockIdx.z;
    const int hl = 4 * blockIdx.x + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    grid_dep_wait();  // the partials of the attention kernel launched just before
    if (hl >= NH) return;
    // the partials of (row t, head group hg): its splits, or in stream-K mode
    // the CTAs whose unit runs overlap the pair's tiles (slot = 2 CTA + segment)
    const size_t base = ((size_t)t * gridDim.y + hg) * a.splits;
    int64_t c_lo = 0, n_part = a.splits;
    const int64_t U = a.sk_units, Cg = a.sk_ctas / (int64_t)gridDim.y, tpr = a.sk_tpr;
    if (Cg > 0) {
        // head group hg's CTAs share U = T * tpr units; the CTA (within the
        // head group) of unit u is ((u + 1) Cg - 1) / U
        const int64_t u_lo = (int64_t)t * tpr, u_hi = u_lo + tpr - 1;
        c_lo = ((u_lo + 1) * Cg - 1) / U;
        n_part = ((u_hi + 1) * Cg - 1) / U - c_lo + 1;
    }
    float M = -CUDART_INF_F, L = 0.0f;
    float4 acc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
    for (int s = 0; s < n_part; ++s) {
        size_t slot;
        if (Cg > 0) {
            const int64_t c = c_lo + s, cta = hg * Cg + c;
            slot = (size_t)(2 * cta + ((c * U / Cg) / tpr == t ? 0 : 1)) * kHG + hl;
        } else {
            slot = (base + s) * kHG + hl;
        }
        const float m = __ldcg(a.part_ml + slot * 2), l = __ldcg(a.part_ml + slot * 2 + 1);
        const float4 *src = reinterpret_cast<const float4 *>(a.part_o + slot * kDv) + lane;
        float4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = __ldcg(src + 32 * k);
        if (l > 0.0f) {
            const float Mn = fmaxf(M, m);
            const float cs = M == -CUDART_INF_F ? 0.0f : exp2f(M - Mn), cn = exp2f(m - Mn);
            L = L * cs + l * cn;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                acc[k].x = acc[k].x * cs + v[k].x * cn;
                acc[k].y = acc[k].y * cs + v[k].y * cn;
                acc[k].z = acc[k].z * cs + v[k].z * cn;
                acc[k].w = acc[k].w * cs + v[k].w * cn;
            }
            M = Mn;
        }
    }
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
    uint2 *o = reinterpret_cast<uint2 *>(a.out + ((size_t)t * a.H + hg * NH + hl) * kDv) + lane;
#pragma unroll
    for (int k = 0; k < 4; ++k)
        o[32 * k] = make_uint2(pack_bf16(acc[k].x * inv, acc[k].y * inv), pack_bf16(acc[k].z * inv, acc[k].w * inv));
    if (a.lse && lane == 0)
        a.lse[(size_t)t * a.H + hg * NH + hl] = L > 0.0f ? M * 0.69314718055994531f + logf(L) : -CUDART_INF_F;
}

}  // namespace

size_t mla_smem_bytes(int NH) {
    (void)NH;
    return 1024 + (size_t)MlaLayout<64>::kMiscOff + sizeof(MlaBars) + sizeof(MlaStats);
}
int mla_key_tile() { return kKeys; }

template <int NH, bool kPair, bool kF8, bool kSK = false>
static cudaError_t launch_tc(const CUtensorMap &tq, const MlaArgs &a, cudaStream_t st) {
    const size_t smem = mla_smem_bytes(NH);
    auto kern = sparse_mla_tc_kernel<NH, kPair, kF8, kSK>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = kSK ? dim3((unsigned)a.sk_ctas, 1, 1) : dim3((unsigned)(a.H / NH), (unsigned)a.splits, (unsigned)a.T);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kPair ? 2 : 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, tq, a);
}

template <bool kF8>
static cudaError_t launch_heads(const CUtensorMap &tq, const MlaArgs &a, int NH, bool pair, cudaStream_t st) {
    if (NH == 64 && a.sk_ctas > 0 && !pair) return launch_tc<64, false, kF8, true>(tq, a, st);
    if (NH == 64 && a.H == 128 && pair) return launch_tc<64, true, kF8>(tq, a, st);
    if (NH == 64) return launch_tc<64, false, kF8>(tq, a, st);
    if (NH == 32) return launch_tc<32, false, kF8>(tq, a, st);
    if (NH == 16) return launch_tc<16, false, kF8>(tq, a, st);
    return cudaErrorInvalidValue;
}

cudaError_t launch_mla_combine(const MlaArgs &a, int NH, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((NH + 3) / 4, a.H / NH, a.T);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, mla_combine_kernel, a, NH);
}

cudaError_t launch_sparse_mla(const CUtensorMap &tq, const MlaArgs &a, int NH, bool fp8, bool pair, cudaStream_t st) {
    const cudaError_t e = fp8 ? launch_heads<true>(tq, a, NH, pair, st) : launch_heads<false>(tq, a, NH, pair, st);
    if (e != cudaSuccess || (a.splits == 1 && a.sk_ctas == 0)) return e;
    return launch_mla_combine(a, NH, st);
}

}  // namespace dsa
