// sparse_mla_ds.cu -- sparse MLA for 128-head queries, with the 576 latent
// dims of every selected row split between the two CTAs of a cluster.
//
// What it computes is the same as sparse_mla.cu ("Day0 Inference Support and
// Performance Optimization for New-Architecture LLMs", §2 item 2 and §4
// "Sparse attention reads by index"; "Day0 Inference Optimization for a New
// Hybrid Attention Architecture: A Full-Stack Deep Dive", operator fusion
// item 1): for query row t and head h,
//     out[t][h] = sum_i softmax_i(scale * q[t][h] . kv[idx_i]) * kv[idx_i][0:512]
// over the valid selected positions idx_i of row t.
//
// Design.  One cluster of two CTAs takes one (query row, key split) with all
// 128 heads.  CTA r owns the latent dims 256 r .. 256 r + 255 (four 64-dim
// regions) and the rope dims 512 + 32 r .. 512 + 32 r + 31 (one region of
// 64-byte rows).  Each CTA gathers only its dims of every selected row (36 KB
// per 64-key tile), so each row is read from memory once.  Per tile:
//   logits   S_r[128 heads x 64 keys] = Q[:, dims_r] . K_tile[:, dims_r]^T
//            (M = 128: every head in one MMA; the latent part of Q sits in
//            TMEM as the A operand, its rope part in shared memory);
//   exchange the exchange warps send S_r (fp32, 32 KB) to the other CTA with
//            st.async over distributed shared memory while the softmax warps
//            work on the previous tile (two logits buffers in TMEM, two
//            receive buffers in shared memory);
//   softmax  both CTAs add the two partials -- the same fp32 sums in both,
//            addition commutes -- and run the same online softmax, so their
//            P, running max and sum agree bit for bit; the receive buffer is
//            handed back to the other CTA as soon as it has been read;
//   P.V      O_r^T[256 dims x 128 heads] += V_tile[:, dims_r]^T . P^T (two
//            M = 128 chunks of value dims, N = 128 heads), V read MN-major
//            from the gathered tile; O^T keeps value dims in TMEM lanes, so
//            the epilogue's stores are coalesced along dims.
// TMEM (512 columns): O^T 0..255 (chunk c at 128 c), S buffers 256 and 320,
// the latent part of Q 384..511.
// Warps: 0-3 gather (cp.async into 128-byte-swizzled regions), 4 tcgen05
// issuer, 5-8 exchange, 9-12 softmax (warp w reads TMEM lanes 32 (w % 4) ..);
// warps 5-12 run the epilogue.  Tiles whose 64 index slots hold no valid
// position (the -1 padding of rows with fewer than K candidates) are skipped:
// both CTAs build the same list of the others from the same row table.  Key splits write the partial layout of
// sparse_mla.cu and are merged by its combine kernel.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "ptx.cuh"
#include "kernels.h"

namespace dsa {

namespace {

constexpr int kD = 576;
constexpr int kDv = 512;
constexpr int kHeads = 128;
constexpr int kKeys = 64;                       // keys per tile (N of the logits MMA)
constexpr int kRegionBytes = kKeys * 128;       // 64 keys x 64 dims, bf16, 128-byte rows
constexpr int kRopeBytes = kKeys * 64;          // this CTA's 32 rope dims, 64-byte rows
constexpr int kStageBytes = 4 * kRegionBytes + kRopeBytes;
constexpr int kStages = 3;
constexpr int kGather = 4;                      // gather warps
constexpr int kMmaWarp = kGather;
constexpr int kXWarp0 = kGather + 1;            // 4 exchange warps
constexpr int kSmWarp0 = kXWarp0 + 4;           // 4 softmax warps
constexpr int kThreads = (kSmWarp0 + 4) * 32;
constexpr int kBarGather = 2, kBarSm = 3, kBarEpi = 4;
constexpr int kMaxKeys = 2048;                  // keys of one split, at most (host keeps this)
constexpr int kXBytes = kHeads * kKeys * 4;     // one partial logits tile, fp32
constexpr uint32_t kColO = 0, kColS = 256, kColQ = 384;

constexpr int kPBytes = kHeads * kKeys * 2;     // P^T of one tile, bf16
constexpr int kXOff = kStages * kStageBytes;    // two receive buffers (1024-aligned)
constexpr int kPOff = kXOff + 2 * kXBytes;      // two P^T buffers
constexpr int kQrOff = kPOff + 2 * kPBytes;     // this CTA's rope dims of Q, [128 heads][32 dims]
constexpr int kBarOff = kQrOff + kHeads * 64;
static_assert(kStageBytes % 1024 == 0 && kXOff % 1024 == 0 && kPOff % 1024 == 0 && kQrOff % 1024 == 0,
              "swizzled operands start on 1024-byte boundaries");

struct __align__(16) DsBars {
    uint64_t kv_full[kStages], kv_empty[kStages];
    uint64_t s_full[2], s_free[2];
    uint64_t x_full[2];   // the other CTA's partial logits for this buffer have landed here
    uint64_t x_free[2];   // the other CTA's receive buffer may take the next tile
    uint64_t q_full, p_full, o_done, o_full, drain, table;
    uint32_t tmem_slot;
    int abort[2];  // [0] a wait gave up; [1] wait limit in microseconds (0: default)
};

struct __align__(16) DsTable {
    int32_t rows[kMaxKeys];            // physical cache row of every key of the split
    uint32_t valid[kMaxKeys / 32];     // bit k % 32 of word k / 32: key k is valid
    float alpha[kHeads];               // this tile's rescale factor per head
    float m_fin[kHeads], l_fin[kHeads], inv_l[kHeads];
    int32_t tile_list[kMaxKeys / kKeys];  // the split's tiles that hold a valid key, in order
    int32_t n_work;                       // their number
};

__device__ __forceinline__ int find_seq(const int32_t *cu_q, int B, int t) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(cu_q + mid) <= t) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
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

__global__ void __launch_bounds__(kThreads, 1) sparse_mla_ds_kernel(MlaArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sKV = smem;
    uint8_t *sX = smem + kXOff;    // receive buffer j at j * kXBytes: [16 chunks][128 heads] float4
    uint8_t *sP = smem + kPOff;    // P^T buffer j at j * kPBytes
    uint8_t *sQr = smem + kQrOff;
    DsBars *bars = reinterpret_cast<DsBars *>(smem + kBarOff);
    DsTable *tab = reinterpret_cast<DsTable *>(bars + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank(), peer = rank ^ 1u;
    const int t = blockIdx.z;
    const int k_begin = blockIdx.y * a.keys_per_split;
    const int k_end = min(a.K, k_begin + a.keys_per_split);
    const int n_tiles = k_end > k_begin ? (k_end - k_begin + kKeys - 1) / kKeys : 0;
    // Inputs may come from the kernel launched just before this one (the
    // indexer's indices); with programmatic dependent launch this kernel
    // starts early and waits here until they are visible.
    grid_dep_wait();
    const int b = find_seq(a.cu_q, a.B, t);
    const int pos = __ldg(a.seq_lens + b) - (__ldg(a.cu_q + b + 1) - __ldg(a.cu_q + b)) + (t - __ldg(a.cu_q + b));

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&bars->kv_full[i], 32 * kGather);  // one cp.async completion arrival per gather lane
            mbar_init(&bars->kv_empty[i], 1);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(&bars->s_full[j], 1);
            mbar_init(&bars->s_free[j], 8);   // exchange and softmax warps have read the logits
            mbar_init(&bars->x_full[j], 1);
            mbar_init(&bars->x_free[j], 1);   // one remote arrival from the other CTA
        }
        mbar_init(&bars->q_full, 4);
        mbar_init(&bars->p_full, 4);
        mbar_init(&bars->o_done, 1);
        mbar_init(&bars->o_full, 1);
        mbar_init(&bars->drain, 1);
        mbar_init(&bars->table, 1);
        bars->abort[0] = 0;
        bars->abort[1] = wait_limit_us(a.err);
        fence_mbar_init();
        // the receive buffers expect tiles 0 and 1 (bytes may land from the
        // cluster barrier below on)
        for (int j = 0; j < 2 && j < n_tiles; ++j) mbar_arrive_expect_tx(&bars->x_full[j], kXBytes);
    }
    if (warp == kMmaWarp) tmem_alloc(&bars->tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_barrier();  // both CTAs' barriers are initialised before any remote arrival or store
    const uint32_t tmem = bars->tmem_slot;
    volatile int *abort = bars->abort;
    const int wl = abort[1];  // test wait limit in microseconds (0: the default limit)

    if (warp < kGather) {
        // ---------------------------------------------------------------- gather
        // resolve every selected key of the split to its physical row once
        const int n_keys = n_tiles * kKeys;
        constexpr int kPer = kMaxKeys / (kGather * 32);
        int idxv[kPer], pagev[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int k = threadIdx.x + u * kGather * 32, slot = k_begin + k;
            idxv[u] = k < n_keys && slot < a.K ? __ldg(a.indices + (size_t)t * a.K + slot) : -1;
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u)
            pagev[u] = idxv[u] >= 0 && idxv[u] <= pos && idxv[u] / a.page_size < a.max_pages
                           ? __ldg(a.page_table + (size_t)b * a.max_pages + idxv[u] / a.page_size)
                           : -1;
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int k = threadIdx.x + u * kGather * 32;
            if (k >= n_keys) break;  // n_keys is a multiple of 64: warp-uniform
            const int idx = idxv[u];
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
            tab->rows[k] = row;
            const uint32_t bits = __ballot_sync(0xffffffffu, v);
            if (lane == 0) tab->valid[k >> 5] = bits;
        }
        bar_sync(kBarGather, kGather * 32);
        // the tiles with at least one valid key (at most 32 per split)
        if (warp == 0) {
            const bool any = lane < n_tiles && (tab->valid[2 * lane] | tab->valid[2 * lane + 1]) != 0u;
            const uint32_t mask = __ballot_sync(0xffffffffu, any);
            if (any) tab->tile_list[__popc(mask & ((1u << lane) - 1u))] = lane;
            if (lane == 0) tab->n_work = __popc(mask);
        }
        bar_sync(kBarGather, kGather * 32);
        if (threadIdx.x == 0) mbar_arrive(&bars->table);
        const int n_work = tab->n_work;
        // warp w: keys 16 w .. 16 w + 15.  Latent regions: lane l copies chunk
        // l % 8 of keys 16 w + l / 8 + 4 m; rope: chunk l % 4 of this rank's
        // 64-byte half of keys 16 w + l / 4 + 8 m
        const int kl = warp * 16 + (lane >> 3), cl = lane & 7;
        const int kr = warp * 16 + (lane >> 2), cr = lane & 3;
        const uint8_t *src_l = a.kv + 512 * rank + cl * 16;  // + row * 1152 + region * 128
        const uint8_t *src_r = a.kv + 1024 + 64 * rank + cr * 16;
        for (int i = 0; i < n_work; ++i) {
            const int stg = i % kStages;
            bool ok = true;
            if (i >= kStages) ok = mbar_wait(&bars->kv_empty[stg], ((i / kStages) & 1) ^ 1, a.err, 0x601, abort, wl);
            if (!__all_sync(0xffffffffu, ok)) break;
            uint8_t *dst = sKV + stg * kStageBytes;
            const int32_t *rows = tab->rows + tab->tile_list[i] * kKeys;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int key = kl + 4 * m;
                const uint8_t *src = src_l + (size_t)rows[key] * (kD * 2);
                uint8_t *d = dst + key * 128 + ((cl ^ (key & 7)) << 4);
#pragma unroll
                for (int r = 0; r < 4; ++r) cp_async16(d + r * kRegionBytes, src + r * 128);
            }
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const int key = kr + 8 * m;
                cp_async16(dst + 4 * kRegionBytes + key * 64 + ((cr ^ ((key >> 1) & 3)) << 4),
                           src_r + (size_t)rows[key] * (kD * 2));
            }
            cp_async_arrive(&bars->kv_full[stg]);
        }
        cp_async_wait_all();  // the CTA stays alive until every copy has landed
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- tcgen05 issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(kHeads, kKeys);
            constexpr uint32_t idesc_o = idesc_bf16_f32_amn(128, kHeads);  // V^T MN-major, P^T K-major
            const uint32_t kv_base = smem_u32(sKV), p_base = smem_u32(sP), qr_base = smem_u32(sQr);
            bool ok = mbar_wait(&bars->table, 0, a.err, 0x60d, abort, wl);
            const int n_work = tab->n_work;
            ok = ok && n_work > 0 && mbar_wait(&bars->q_full, 0, a.err, 0x602, abort, wl);
            // logits of tile i into S buffer i & 1: its four latent regions
            // (A = Q in TMEM) and this CTA's two rope steps (A = Q in smem)
            auto ready_s = [&](int i) {
                return mbar_try_wait(&bars->kv_full[i % kStages], (i / kStages) & 1) &&
                       (i < 2 || mbar_try_wait(&bars->s_free[i & 1], ((i - 2) >> 1) & 1));
            };
            auto issue_s = [&](int i) -> bool {
                const int st = i % kStages, sb = i & 1;
                if (!mbar_wait(&bars->kv_full[st], (i / kStages) & 1, a.err, 0x603, abort, wl)) return false;
                if (i >= 2 && !mbar_wait(&bars->s_free[sb], ((i - 2) >> 1) & 1, a.err, 0x604, abort, wl)) return false;
                fence_proxy_async_smem();  // the tile was written through the generic proxy
                tc_fence_after();
                const uint32_t kb = kv_base + st * kStageBytes, d = tmem + kColS + kKeys * sb;
#pragma unroll
                for (int r = 0; r < 4; ++r) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16_ts(d, tmem + kColQ + 32 * r + 8 * kk,
                                    sdesc_kmajor_sw128(kb + r * kRegionBytes + kk * 32), idesc_s, (r | kk) ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
                    mma_bf16_ss(d, sdesc_kmajor_sw64(qr_base + kk * 32), sdesc_kmajor_sw64(kb + 4 * kRegionBytes + kk * 32),
                                idesc_s, 1u);
                mma_commit(&bars->s_full[sb]);
                return true;
            };
            if (ok) ok = issue_s(0);
            if (ok && n_work > 1) ok = issue_s(1);
            for (int i = 0; ok && i < n_work; ++i) {
                // the logits two tiles ahead go first when they can start now
                bool pend = i + 2 < n_work;
                if (pend && ready_s(i + 2)) {
                    if (!(ok = issue_s(i + 2))) break;
                    pend = false;
                }
                if (!(ok = mbar_wait(&bars->p_full, i & 1, a.err, 0x605, abort, wl))) break;
                tc_fence_after();
                // O^T chunk c (value dims 128 c ..) += V^T . P^T
                const uint32_t kb = kv_base + (i % kStages) * kStageBytes, pb = p_base + (i & 1) * kPBytes;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
#pragma unroll
                    for (int j = 0; j < kKeys / 16; ++j)
                        mma_bf16_ss(tmem + kColO + 128 * c,
                                    sdesc_mnmajor_sw128(kb + 2 * c * kRegionBytes + j * 2048, kRegionBytes, 1024),
                                    sdesc_kmajor_sw128(pb + j * 32), idesc_o, (i > 0 || j > 0) ? 1u : 0u);
                }
                mma_commit(&bars->kv_empty[i % kStages]);
                mma_commit(&bars->o_done);
                if (pend && !(ok = issue_s(i + 2))) break;
            }
            if (ok && n_work > 0) mma_commit(&bars->o_full);
            if (*abort) {
                volatile int no_abort[2] = {0, 0};
                mma_commit(&bars->drain);
                mbar_wait(&bars->drain, 0, nullptr, 0, no_abort);
            }
        }
    } else {
        const int quad = warp & 3;
        const bool is_sm = warp >= kSmWarp0;
        const int tid_s = (warp - kSmWarp0) * 32 + lane;  // softmax threads: 0..127
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const uint32_t tl = tmem + lane_off;  // this warp's TMEM lanes
        const int h = quad * 32 + lane;       // head (S rows) or value dim (O^T rows) of this thread
        bool ok = true;
        int n_work = 0;  // tiles with a valid key (known once the row table is built)
        if (!is_sm) {
            // ---------------------------------------------------------------- exchange
            const uint32_t x_peer = map_peer(smem_u32(sX), peer);
            const uint32_t x_full_peer = map_peer(smem_u32(&bars->x_full[0]), peer);
            ok = __all_sync(0xffffffffu, mbar_wait(&bars->table, 0, a.err, 0x60e, abort, wl));
            n_work = ok ? tab->n_work : 0;
            for (int i = 0; i < n_work; ++i) {
                const int sb = i & 1;
                ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[sb], (i >> 1) & 1, a.err, 0x607, abort, wl));
                if (!ok) break;
                tc_fence_after();
                uint32_t s0[32], s1[32];
                tmem_ld32(tl + kColS + kKeys * sb, s0);
                tmem_ld32(tl + kColS + kKeys * sb + 32, s1);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->s_free[sb]);
                // the other CTA's buffer sb is free once it has read tile i - 2
                if (i >= 2)
                    ok = __all_sync(0xffffffffu,
                                    mbar_wait<true>(&bars->x_free[sb], ((i - 2) >> 1) & 1, a.err, 0x608, abort, wl));
                if (!ok) break;
                const uint32_t dst = x_peer + sb * kXBytes + h * 16, bar = x_full_peer + sb * 8;
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    st_async_peer16(dst + q * kHeads * 16, make_uint4(s0[4 * q], s0[4 * q + 1], s0[4 * q + 2], s0[4 * q + 3]),
                                    bar);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    st_async_peer16(dst + (q + 8) * kHeads * 16,
                                    make_uint4(s1[4 * q], s1[4 * q + 1], s1[4 * q + 2], s1[4 * q + 3]), bar);
            }
        } else {
            // ---------------------------------------------------------------- softmax
            // Q: this CTA's latent dims of head h into TMEM (the logits' A
            // operand, row h in lane h), the rope dims into shared memory
            {
                const uint4 *qrow = reinterpret_cast<const uint4 *>(a.q + ((size_t)t * kHeads + h) * kD);
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    uint32_t w[32];
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint4 v = __ldg(qrow + (4 * (int)rank + r) * 8 + c);
                        w[4 * c] = v.x;
                        w[4 * c + 1] = v.y;
                        w[4 * c + 2] = v.z;
                        w[4 * c + 3] = v.w;
                    }
                    tmem_st32(tl + kColQ + 32 * r, w);
                }
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    *reinterpret_cast<uint4 *>(sQr + h * 64 + ((c ^ ((h >> 1) & 3)) << 4)) = __ldg(qrow + 64 + 4 * (int)rank + c);
                tmem_wait_st();
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->q_full);
            }
            const uint32_t x_free_peer = map_peer(smem_u32(&bars->x_free[0]), peer);
            float m_ref = -CUDART_INF_F, l_run = 0.0f;
            int next0 = 0, next1 = 1;  // the tile each receive buffer expects next
            // (decisions to go on are taken by all four softmax warps together,
            // since they meet at named barriers inside the loop)
            ok = bar_and(kBarSm, 128, mbar_wait(&bars->table, 0, a.err, 0x606, abort, wl));
            n_work = ok ? tab->n_work : 0;
            for (int i = 0; ok && i < n_work; ++i) {
                const int sb = i & 1;
                const uint8_t *xb = sX + sb * kXBytes;
                // This CTA's partial logits are read (and their TMEM buffer
                // handed back to the MMA) as soon as they are ready, before
                // the other CTA's partial has landed: the logits of tile
                // i + 2 can then start during the exchange of tile i.
                ok = bar_and(kBarSm, 128, mbar_wait(&bars->s_full[sb], (i >> 1) & 1, a.err, 0x60a, abort, wl));
                if (!ok) break;
                tc_fence_after();
                float s[kKeys];
                {
                    uint32_t r[32];
                    tmem_ld32(tl + kColS + kKeys * sb, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) s[j] = __uint_as_float(r[j]);
                    tmem_ld32(tl + kColS + kKeys * sb + 32, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) s[32 + j] = __uint_as_float(r[j]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->s_free[sb]);
                ok = bar_and(kBarSm, 128, mbar_wait<true>(&bars->x_full[sb], (i >> 1) & 1, a.err, 0x609, abort, wl));
                if (!ok) break;
                // full logits: this CTA's partial plus the other's
#pragma unroll
                for (int q = 0; q < kKeys / 4; ++q) {
                    const float4 v = *reinterpret_cast<const float4 *>(xb + (q * kHeads + h) * 16);
                    s[4 * q] += v.x;
                    s[4 * q + 1] += v.y;
                    s[4 * q + 2] += v.z;
                    s[4 * q + 3] += v.w;
                }
                // every softmax thread has read buffer sb: it expects tile i + 2's
                // partial logits next, and the other CTA may send them
                bar_sync(kBarSm, 128);
                if (tid_s == 0 && i + 2 < n_work) {
                    mbar_arrive_expect_tx(&bars->x_full[sb], kXBytes);
                    mbar_arrive_remote(x_free_peer + sb * 8);
                }
                if (sb) next1 = i + 2;
                else next0 = i + 2;
                // online softmax of head h over the tile's keys (log2 domain);
                // the reference max moves only when the max grows by more than 2^8
                const int tile = tab->tile_list[i];
                const uint32_t v0 = tab->valid[2 * tile], v1 = tab->valid[2 * tile + 1];
                float m4[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
                for (int j = 0; j < kKeys; ++j) {
                    const bool valid = (((j < 32 ? v0 : v1) >> (j & 31)) & 1u) != 0;
                    s[j] = valid ? s[j] * a.scale_log2 : -CUDART_INF_F;
                    m4[j & 3] = fmaxf(m4[j & 3], s[j]);
                }
                const float mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                float al = 1.0f;
                if (mt != -CUDART_INF_F && (m_ref == -CUDART_INF_F || mt > m_ref + 8.0f)) {
                    al = m_ref == -CUDART_INF_F ? 1.0f : exp2f(m_ref - mt);
                    m_ref = mt;
                }
                const float ref = m_ref == -CUDART_INF_F ? 0.0f : m_ref;
                float s4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                uint32_t pw[kKeys / 2];
#pragma unroll
                for (int j = 0; j < kKeys / 2; ++j) {
                    const float p0 = exp2f(s[2 * j] - ref), p1 = exp2f(s[2 * j + 1] - ref);
                    s4[(2 * j) & 3] += p0;
                    s4[(2 * j + 1) & 3] += p1;
                    pw[j] = pack_bf16(p0, p1);
                }
                l_run = l_run * al + ((s4[0] + s4[1]) + (s4[2] + s4[3]));
                tab->alpha[h] = al;
                // P^T as K-major [head][key] rows of 128 bytes, 128-byte swizzle
                // (buffer sb: tile i - 2's P.V has completed)
                uint8_t *pb = sP + sb * kPBytes;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4 *>(pb + h * 128 + ((c ^ (h & 7)) << 4)) =
                        make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
                // the previous tile's P.V must be complete before O^T is rescaled
                ok = bar_and(kBarSm, 128, i == 0 || mbar_wait(&bars->o_done, (i - 1) & 1, a.err, 0x60b, abort, wl));
                if (!ok) break;
                tc_fence_after();
                if (bar_or(kBarSm, 128, al != 1.0f) && i > 0) {
                    // rescale O^T column h by alpha[h] in this warp's 32 value-dim
                    // lanes of both chunks (a rare path)
#pragma unroll 1
                    for (int cc = 0; cc < 16; ++cc) {
                        const uint32_t ta = tl + kColO + 16 * cc;
                        uint32_t o[16];
                        tmem_ld16(ta, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            o[j] = __float_as_uint(__uint_as_float(o[j]) * tab->alpha[(16 * cc + j) & 127]);
                        tmem_st16(ta, o);
                    }
                    tmem_wait_st();
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->p_full);
            }
            tab->m_fin[h] = m_ref;
            tab->l_fin[h] = l_run;
            tab->inv_l[h] = l_run > 0.0f ? 1.0f / l_run : 0.0f;
            if (*abort && tid_s == 0) {
                // The other CTA sends a tile into buffer j once this CTA has
                // freed it: let bytes that may be on their way land (or the
                // bounded wait run out) before this CTA can leave.
                volatile int no_abort[2] = {0, 0};
                if (next0 < n_work) mbar_wait<true>(&bars->x_full[0], (next0 >> 1) & 1, nullptr, 0, no_abort);
                if (next1 < n_work) mbar_wait<true>(&bars->x_full[1], (next1 >> 1) & 1, nullptr, 0, no_abort);
            }
        }
        // ---------------------------------------------------------------- epilogue
        if (tid_s == 0) grid_dep_launch();  // the split combine may start launching
        if (ok && n_work > 0) ok = mbar_wait(&bars->o_full, 0, a.err, 0x60c, abort, wl);
        ok = bar_and(kBarEpi, 256, ok && !*abort);  // also: m_fin / l_fin are written
        tc_fence_after();
        if (ok) {
            const bool direct = a.splits == 1;
            const int c = is_sm ? 0 : 1;                       // value-dim chunk of this warp group
            const int dim = 256 * (int)rank + 128 * c + h;     // this thread's value dim
#pragma unroll 1
            for (int h0 = 0; h0 < kHeads; h0 += 32) {
                uint32_t o[32];
                if (n_work > 0) {
                    tmem_ld32(tl + kColO + 128 * c + h0, o);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = 0u;
                }
                // heads h0 .. h0 + 31 sit in consecutive output rows (and
                // consecutive partial slots of one head group)
                if (direct) {
                    uint16_t *op = a.out + ((size_t)t * kHeads + h0) * kDv + dim;
#pragma unroll
                    for (int j = 0; j < 32; ++j, op += kDv)
                        *op = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(o[j]) * tab->inv_l[h0 + j]));
                } else {
                    float *op = a.part_o + ((((size_t)t * 2 + (h0 >> 6)) * a.splits + blockIdx.y) * 64 + (h0 & 63)) * kDv + dim;
#pragma unroll
                    for (int j = 0; j < 32; ++j, op += kDv) *op = __uint_as_float(o[j]);
                }
            }
            if (rank == 0 && is_sm) {
                // both CTAs hold the same running max and sum; rank 0 writes them
                const float m = tab->m_fin[h], l = tab->l_fin[h];
                if (direct) {
                    if (a.lse)
                        a.lse[(size_t)t * kHeads + h] = l > 0.0f ? m * 0.69314718055994531f + logf(l) : -CUDART_INF_F;
                } else {
                    const size_t slot = (((size_t)t * 2 + (h >> 6)) * a.splits + blockIdx.y) * 64 + (h & 63);
                    a.part_ml[slot * 2 + 0] = l > 0.0f ? m : -CUDART_INF_F;
                    a.part_ml[slot * 2 + 1] = l;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
    // neither CTA leaves while the other may still store into or signal it
    cluster_barrier();
}

}  // namespace

size_t mla_ds_smem_bytes() { return 1024 + (size_t)kBarOff + sizeof(DsBars) + sizeof(DsTable); }

cudaError_t launch_sparse_mla_ds(const MlaArgs &a, cudaStream_t st) {
    if (a.H != kHeads || a.keys_per_split % kKeys != 0 || a.keys_per_split > kMaxKeys) return cudaErrorInvalidValue;
    const size_t smem = mla_ds_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(sparse_mla_ds_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, (unsigned)a.splits, (unsigned)a.T);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, sparse_mla_ds_kernel, a);
    if (e != cudaSuccess || a.splits == 1) return e;
    return launch_mla_combine(a, 64, st);
}

}  // namespace dsa
