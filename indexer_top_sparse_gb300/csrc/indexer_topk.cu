// indexer_topk.cu -- fused lightweight indexer + Top-K for sm_103a.
//
// What it computes ("Optimizing Inference for Hybrid Attention LLMs: A
// Practical Guide to Day-0 Adaptation", §3.1 Indexer Fusion; "Day0 Inference
// Support and Performance Optimization for New-Architecture LLMs", §4 item 1):
// for every query row t and causal position s <= pos(t)
//     score(t, s) = sum_j w[t][j] * ReLU(q_idx[t][j] . k_idx[s])
// then the top K positions by (score desc, position asc).  Scoring, head
// weighting and selection are one kernel; the paged index-key cache is read
// directly; scores stay in shared memory and only indices are written.
//
// Design (one thread-block cluster of C CTAs per group of G query rows of one
// sequence; the group's causal history is split into C contiguous ranges of
// 128-position tiles, one per CTA):
//   warp 0      TMA producer: the group's Q rows once, then per tile two
//               64-row page boxes x two 64-column halves, 128-byte swizzle,
//               into a STAGES-deep ring.
//   warps 1, 6  tcgen05 issuers (even and odd tiles): D[128 pos x 64G] =
//               K_tile[128 x 128] * Q[64G x 128]^T, eight K=16 steps, fp32
//               accumulators in TMEM (one per issuer), commits release the
//               smem stage and hand the TMEM buffer to the epilogue.
//   warps 2-5   epilogue: thread = TMEM lane = position; ReLU, weight by w and
//               sum over the 64 heads in registers; store an order-preserving
//               32-bit key per (query, position) in shared memory.
//   warps 7-11  (one query row per cluster) the selection only.
//   all warps   cluster radix select (8-bit digits, histograms summed across
//               the cluster through distributed shared memory), ties resolved
//               to the lowest positions, indices written in ascending order.
#include <cooperative_groups.h>

#include "ptx.cuh"
#include "kernels.h"
#include "mxfp8.cuh"

namespace cg = cooperative_groups;

namespace dsa {

namespace {

constexpr int kHI = 64;          // index heads
constexpr int kDI = 128;         // index head dim
constexpr int kTileM = 128;      // positions per tile (MMA M)
constexpr int kBox = 64;         // rows / columns per TMA box
constexpr int kBoxBytes = kBox * kBox * 2;           // 8 KB
constexpr int kTileBytes = kTileM * kDI * 2;         // 32 KB
constexpr int kRegionBytes = kTileM * 128;           // one 64-column half of a tile: 16 KB
constexpr int kThreads = 192;    // score-row selection kernel
// The bf16 indexer: warp 0 TMA, warps 1 and 6 tcgen05 issue (even and odd
// tiles), warps 2..5 epilogue.  One thread's waits, MMA issues and commits
// for a tile take longer than the tensor core needs for it, so two threads
// issue alternate tiles; the ring depth is even, so each stage is always
// filled for and consumed by the same thread, whose waits on its barriers
// therefore come in phase order.  With one query row per cluster (decode) five more
// warps join only the selection, whose passes over the keys are bound by
// latency at two warps per scheduler; the wider epilogue registers of
// several rows leave no room for them.
template <int G>
constexpr int idx_threads() { return G == 1 ? 384 : 224; }
constexpr int kIdxIssuer2 = 6;
constexpr int kHist = 256;
constexpr int kMaxCluster = 16;

// Order-preserving map from a finite float to uint32 (larger float -> larger
// key); -0 is folded onto +0.  Every finite value maps above 0x007FFFFF, so 0
// marks "not a candidate".
__device__ __forceinline__ uint32_t score_key(float x) {
    uint32_t u = __float_as_uint(x == 0.0f ? 0.0f : x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int kCandCap = 128;   // threshold-bucket keys one CTA may hand to the bucket selection
constexpr int kAllCap = 512;    // the same for the whole cluster
constexpr int kMaxSelThreads = 384;

// Shared state of the cluster selection for up to kSegMax threads per CTA.
template <int kSegMax>
struct __align__(16) SelectSmemT {
    uint32_t hist[2][kHist];
    uint32_t tot[kHist];
    int32_t scan[2][kSegMax / 32 > 16 ? kSegMax / 32 : 16];  // one word per warp
    int32_t cnt[4];       // this CTA's (n_gt, n_eq) for the cluster exchange; [2] = abort flag
    uint32_t bcast[4];    // digit, count-above
    // bucket selection: published [keys above the bucket, bucket keys kept, overflow, pos0]
    int32_t pub[4];
    uint32_t ncand;
    uint32_t pad_[3];
    uint32_t cand_key[kCandCap];
    int32_t cand_loc[kCandCap];
    uint32_t all_key[kAllCap];
    int32_t all_pos[kAllCap];
    int32_t all_cta[kAllCap];
    int32_t cta_off[kMaxCluster + 1];
    int32_t cta_pos0[kMaxCluster];  // first position of each CTA's run
    int32_t cta_gt[kMaxCluster];
    int32_t cta_sel[kMaxCluster];
    int32_t seg_sel[kSegMax];
};
using SelectSmem = SelectSmemT<kMaxSelThreads>;

// Exclusive scan of one int per thread across the CTA (kT threads).
template <int kT>
__device__ __forceinline__ int block_exclusive_scan(int v, int32_t *warp_tot, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    int before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kT / 32; ++w) {
        int t = warp_tot[w];
        if (w < warp) before += t;
        all += t;
    }
    __syncthreads();
    if (total) *total = all;
    return before + x - v;
}

// Warp 0 (lanes = threads 0..31): the 8-bit digit whose bucket of h[256]
// holds the krem-th largest counted key, and the count above that bucket,
// into bcast[0], bcast[1] (left as they are if the counts add up to fewer
// than krem).
__device__ __forceinline__ void digit_from_top_warp(const uint32_t *h, int krem, uint32_t *bcast) {
    const int lane = threadIdx.x & 31;
    // digits from high to low: lane L owns digits 255-8L .. 248-8L
    uint32_t part = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) part += h[255 - 8 * lane - i];
    uint32_t incl = part;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    uint32_t excl = incl - part;
    bool mine = excl < (uint32_t)krem && (uint32_t)krem <= incl;
    unsigned ball = __ballot_sync(0xffffffffu, mine);
    int src = __ffs(ball) - 1;
    if (lane == src) {
        uint32_t above = excl;
        int digit = 255 - 8 * lane;
        for (int i = 0; i < 8; ++i, --digit) {
            uint32_t c = h[digit];
            if (above + c >= (uint32_t)krem) break;
            above += c;
        }
        bcast[0] = (uint32_t)digit;
        bcast[1] = above;
    }
}

// Final step of the selection once two radix digits have fixed the top 16
// bits of the threshold (prefix under mask) and krem keys are still needed
// from that 16-bit bucket, which typically holds a few dozen keys: every CTA
// counts its keys above the bucket per thread segment and lists its bucket
// keys; all CTAs copy the cluster's list and rank it by (key descending,
// position ascending), mark their own bucket keys selected (all ones) or not
// (zero) in place, and write their selected positions in order after those
// of the lower-ranked CTAs.  Returns false, with every CTA agreeing, when the
// bucket is too large for this path (the caller continues digit by digit).
template <int kT, class SS>
__device__ bool select_from_bucket(uint32_t kb, int n_local, int pos0, int K, int32_t *out, SS &ss,
                                   uint32_t prefix, uint32_t mask, int krem) {
    static_assert(kT * sizeof(int32_t) <= sizeof(ss.seg_sel), "segment counters");
    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks(), my = (int)cluster.block_rank();
    const int tid = threadIdx.x;
    if (tid == 0) ss.ncand = 0u;
    ss.seg_sel[tid] = 0;
    if (tid < kMaxCluster) ss.cta_sel[tid] = 0;
    __syncthreads();
    // segments of a multiple of four keys, read 16 bytes at a time (the key
    // buffers are 16-byte aligned and readable up to n_local rounded up to 4)
    const int seg = (((n_local + kT - 1) / kT) + 3) & ~3;
    const int l0 = min(n_local, tid * seg), l1 = min(n_local, l0 + seg);
    int n_gt = 0;
    for (int l = l0; l < l1; l += 8) {
        // both 16-byte loads issued before either is used
        const uint4 va = lds128(kb + 4 * l);
        const uint4 vb = l + 4 < l1 ? lds128(kb + 4 * (l + 4)) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t k8[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
        uint32_t eqm = 0u;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const uint32_t m = k8[u] & mask;
            const bool in = l + u < l1 && k8[u] != 0u;
            n_gt += (in && m > prefix) ? 1 : 0;
            eqm |= (in && m == prefix) ? 1u << u : 0u;
        }
        if (eqm != 0u) {
            // (rare) keys in the bucket
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if ((eqm >> u) & 1u) {
                    const uint32_t c = atomicAdd(&ss.ncand, 1u);
                    if (c < (uint32_t)kCandCap) {
                        ss.cand_key[c] = k8[u];
                        ss.cand_loc[c] = l + u;
                    }
                }
            }
        }
    }
    int cta_gt = 0;
    block_exclusive_scan<kT>(n_gt, ss.scan[1], &cta_gt);
    if (tid == 0) {
        ss.pub[0] = cta_gt;
        ss.pub[1] = (int)min(ss.ncand, (uint32_t)kCandCap);
        ss.pub[2] = ss.ncand > (uint32_t)kCandCap;
        ss.pub[3] = pos0;
    }
    cluster.sync();
    if (tid < C) {
        const int4 p = *reinterpret_cast<const int4 *>(cluster.map_shared_rank(ss.pub, tid));
        ss.cta_gt[tid] = p.x;
        ss.cta_off[tid + 1] = p.z ? -1 : p.y;  // -1 marks an overflow
        ss.cta_pos0[tid] = p.w;
    }
    __syncthreads();
    bool fits = true;
    int total = 0;
    for (int c = 0; c < C; ++c) {
        const int n = ss.cta_off[c + 1];
        fits = fits && n >= 0;
        total += max(n, 0);
    }
    fits = fits && total <= kAllCap;
    __syncthreads();
    if (!fits) {
        cluster.sync();  // nobody reuses the shared state another CTA may still read
        return false;
    }
    if (tid == 0) {
        int o = 0;
        for (int c = 0; c < C; ++c) {
            const int n = ss.cta_off[c + 1];
            ss.cta_off[c] = o;
            o += n;
        }
        ss.cta_off[C] = o;
    }
    __syncthreads();
    for (int i = tid; i < total; i += kT) {
        int c = 0;
        while (c + 1 < C && ss.cta_off[c + 1] <= i) ++c;
        const int li = i - ss.cta_off[c];
        const uint32_t k = cluster.map_shared_rank(ss.cand_key, c)[li];
        const int l = cluster.map_shared_rank(ss.cand_loc, c)[li];
        ss.all_key[i] = k;
        ss.all_pos[i] = ss.cta_pos0[c] + l;
        ss.all_cta[i] = c;
    }
    __syncthreads();
    cluster_arrive();  // done reading the other CTAs; the matching wait is at the end
    // Rank the bucket's keys (they share the top 16 bits): one more digit
    // (bits 15..8) takes the keys above its bucket and leaves the rest out;
    // the few keys in it are ranked by (key descending, position ascending).
    // ss.hist[0] is free: the other CTAs read it only before pass 1's barrier.
    uint32_t *h2 = ss.hist[0];
    for (int d = tid; d < kHist; d += kT) h2[d] = 0u;
    if (tid == 0) {
        ss.bcast[0] = 0u;
        ss.bcast[1] = 0u;
    }
    __syncthreads();
    for (int i = tid; i < total; i += kT) red_shared_add(smem_u32(&h2[(ss.all_key[i] >> 8) & 0xFFu]), 1u);
    __syncthreads();
    if (tid < 32) digit_from_top_warp(h2, krem, ss.bcast);
    __syncthreads();
    const uint32_t d2 = ss.bcast[0] & 0xFFu;
    const int krem2 = krem - (int)ss.bcast[1];
    const uint32_t ak = smem_u32(ss.all_key), ap = smem_u32(ss.all_pos);
    for (int i = tid; i < total; i += kT) {
        const uint32_t ki = ss.all_key[i];
        const int pi = ss.all_pos[i];
        bool sel = ((ki >> 8) & 0xFFu) > d2;
        if (((ki >> 8) & 0xFFu) == d2) {
            // (the shared loads are issued eight at a time: each volatile load
            // would otherwise wait for the one before)
            int r = 0, j = 0;
            for (; j + 8 <= total; j += 8) {
                uint32_t kj[8];
                int pj[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) kj[u] = lds32(ak + 4 * (j + u));
#pragma unroll
                for (int u = 0; u < 8; ++u) pj[u] = (int)lds32(ap + 4 * (j + u));
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    r += ((kj[u] >> 8) & 0xFFu) == d2 && ((kj[u] > ki) || (kj[u] == ki && pj[u] < pi));
            }
            for (; j < total; ++j) {
                const uint32_t kj = lds32(ak + 4 * j);
                const int pj = (int)lds32(ap + 4 * j);
                r += ((kj >> 8) & 0xFFu) == d2 && ((kj > ki) || (kj == ki && pj < pi));
            }
            sel = r < krem2;
        }
        const int c = ss.all_cta[i];
        ss.all_cta[i] = c | (sel ? 0x10000 : 0);  // (no other thread reads entry i)
        if (c == my) {
            const int l = pi - pos0;
            sts32(kb + 4 * l, sel ? 0xFFFFFFFFu : 0u);
            if (sel) atomicAdd(&ss.seg_sel[l / seg], 1);
        }
    }
    __syncthreads();
    // selected candidates of each CTA (its candidates are one run of the list)
    {
        const int warp = tid >> 5, lane = tid & 31;
        for (int c = warp; c < C; c += kT / 32) {
            int n = 0;
            for (int i = ss.cta_off[c] + lane; i < ss.cta_off[c + 1]; i += 32) n += ss.all_cta[i] >> 16;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
            if (lane == 0) ss.cta_sel[c] = n;
        }
    }
    __syncthreads();
    int base = 0;
    for (int c = 0; c < my; ++c) base += ss.cta_gt[c] + ss.cta_sel[c];
    int slot = base + block_exclusive_scan<kT>(n_gt + ss.seg_sel[tid], ss.scan[0], nullptr);
    for (int l = l0; l < l1; l += 8) {
        const uint4 va = lds128(kb + 4 * l);
        const uint4 vb = l + 4 < l1 ? lds128(kb + 4 * (l + 4)) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t k8[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (l + u < l1 && k8[u] != 0u && (k8[u] & mask) > prefix && slot < K) out[slot++] = pos0 + l + u;
    }
    cluster_wait();  // nobody leaves while another CTA may still read its candidates
    return true;
}

// Cluster-wide exact Top-K over keys held in shared memory.
//   keys[0..n_local)   this CTA's keys, for positions pos0 + l (0 = invalid)
//   n_valid            number of valid positions across the whole cluster
// Writes min(K, n_valid) positions in ascending order to out[0..] and -1 to
// the rest of out[0..K).  Every CTA of the cluster must call this with the
// same n_valid and K (it contains cluster barriers).
template <int kT, class SS>
__device__ void cluster_topk(const uint32_t *keys, int n_local, int pos0, int n_valid, int K, int32_t *out,
                             SS &ss, const uint32_t *hist0 = nullptr) {
    cg::cluster_group cluster = cg::this_cluster();
    const unsigned C = cluster.num_blocks();
    const unsigned my = cluster.block_rank();
    const int tid = threadIdx.x;

    if (n_valid <= K) {
        // every valid position is selected; positions are contiguous from 0,
        // so slot == position
        const uint32_t kb = smem_u32(keys);
        for (int l = tid; l < n_local; l += kT) {
            if (lds32(kb + 4 * l) != 0u && pos0 + l < n_valid) out[pos0 + l] = pos0 + l;
        }
        if (my == 0) {
            for (int i = (n_valid > 0 ? n_valid : 0) + tid; i < K; i += kT) out[i] = -1;
        }
        cluster.sync();
        return;
    }

    const uint32_t kb = smem_u32(keys);
    uint32_t prefix = 0, mask = 0;
    int krem = K;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        uint32_t *h = ss.hist[pass & 1];
        if (pass == 0 && hist0 != nullptr) {
            // the top-digit histogram was built while the scores were produced
            for (int d = tid; d < kHist; d += kT) h[d] = hist0[d];
        } else {
            for (int d = tid; d < kHist; d += kT) h[d] = 0u;
            __syncthreads();
            const uint32_t hb = smem_u32(h);
            // eight keys per thread loaded before any count; counts predicated
            int l = tid;
            for (; l + 7 * kT < n_local; l += 8 * kT) {
                uint32_t k8[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) k8[u] = lds32(kb + 4 * (l + u * kT));
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    red_shared_add_if(hb + 4 * ((k8[u] >> shift) & 0xFFu), k8[u] != 0u && (k8[u] & mask) == prefix);
            }
            for (; l < n_local; l += kT) {
                const uint32_t k = lds32(kb + 4 * l);
                red_shared_add_if(hb + 4 * ((k >> shift) & 0xFFu), k != 0u && (k & mask) == prefix);
            }
        }
        cluster.sync();
        for (int d4 = tid; d4 < kHist / 4; d4 += kT) {
            // four bins per thread, four CTAs' loads issued before summing
            uint4 s = make_uint4(0u, 0u, 0u, 0u);
            for (int c0 = 0; c0 < (int)C; c0 += 4) {
                uint4 v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    v[u] = c0 + u < (int)C ? reinterpret_cast<const uint4 *>(cluster.map_shared_rank(h, c0 + u))[d4]
                                           : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    s.x += v[u].x;
                    s.y += v[u].y;
                    s.z += v[u].z;
                    s.w += v[u].w;
                }
            }
            reinterpret_cast<uint4 *>(ss.tot)[d4] = s;
        }
        // digit 0, nothing above it, unless a lane below finds the digit that
        // holds the krem-th key: after an aborted wait the counts may add up
        // to fewer than krem keys, and every CTA must still take the same
        // (deterministic) branch, since the cluster barriers follow from it
        if (tid == 0) {
            ss.bcast[0] = 0u;
            ss.bcast[1] = 0u;
        }
        __syncthreads();
        if (tid < 32) digit_from_top_warp(ss.tot, krem, ss.bcast);
        __syncthreads();
        // (masked: after an aborted wait the counts may not add up)
        const uint32_t digit = ss.bcast[0] & 0xFFu;
        krem -= (int)ss.bcast[1];
        prefix |= digit << shift;
        mask |= 0xFFu << shift;
        const bool done = ss.tot[digit] == (uint32_t)krem;
        __syncthreads();
        if (done) break;
        if (pass == 1 && select_from_bucket<kT>(kb, n_local, pos0, K, out, ss, prefix, mask, krem)) return;
    }

    // count (key > threshold) and (key == threshold) in this CTA, by contiguous
    // segments so that output order follows position order
    const int seg = (n_local + kT - 1) / kT;
    const int l0 = min(n_local, tid * seg), l1 = min(n_local, l0 + seg);
    int n_gt = 0, n_eq = 0;
    for (int l = l0; l < l1; ++l) {
        uint32_t k = lds32(kb + 4 * l);
        if (k == 0u) continue;
        uint32_t m = k & mask;
        n_gt += m > prefix;
        n_eq += m == prefix;
    }
    int cta_gt = 0, cta_eq = 0;
    const int eq_before_seg = block_exclusive_scan<kT>(n_eq, ss.scan[0], &cta_eq);
    const int gt_before_seg = block_exclusive_scan<kT>(n_gt, ss.scan[1], &cta_gt);
    if (tid == 0) {
        ss.cnt[0] = cta_gt;
        ss.cnt[1] = cta_eq;
    }
    cluster.sync();
    int eq_before_cta = 0, out_before_cta = 0;
    {
        int2 rc[kMaxCluster];
#pragma unroll
        for (int c = 0; c < kMaxCluster; ++c)
            rc[c] = c < (int)my ? *reinterpret_cast<const int2 *>(cluster.map_shared_rank(ss.cnt, c)) : make_int2(0, 0);
#pragma unroll
        for (int c = 0; c < kMaxCluster; ++c) {
            const int take = min(max(krem - eq_before_cta, 0), rc[c].y);
            out_before_cta += rc[c].x + take;
            eq_before_cta += rc[c].y;
        }
    }
    // per-segment selection counts, then their exclusive scan
    const int eq_rank0 = eq_before_cta + eq_before_seg;
    const int take_seg = min(max(krem - eq_rank0, 0), n_eq);
    const int sel_before_seg = block_exclusive_scan<kT>(n_gt + take_seg, ss.scan[0], nullptr);
    (void)gt_before_seg;
    int slot = out_before_cta + sel_before_seg, eq_rank = eq_rank0;
    for (int l = l0; l < l1; ++l) {
        uint32_t k = lds32(kb + 4 * l);
        if (k == 0u) continue;
        uint32_t m = k & mask;
        bool sel = m > prefix;
        if (m == prefix) {
            sel = eq_rank < krem;
            ++eq_rank;
        }
        if (sel && slot < K) out[slot++] = pos0 + l;
    }
    // nobody may reuse or leave shared memory another CTA still reads
    cluster.sync();
}

template <int G>
struct IdxLayout {
    static constexpr int kQBytes = G * kHI * kDI * 2;  // both 64-column halves
    static constexpr int kQRegion = G * kHI * 128;     // one half: G*64 rows x 128 B
    static constexpr int kN = G * kHI;                 // MMA N
    static constexpr int kTmemCols = 2 * kN <= 32 ? 32 : (2 * kN <= 64 ? 64 : (2 * kN <= 128 ? 128 : (2 * kN <= 256 ? 256 : 512)));
};

struct __align__(16) IdxBars {
    uint64_t drain[2];  // one per issuing thread
    uint64_t full[8];
    uint64_t empty[8];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t qbar;
    uint32_t tmem_slot;
    int abort[2];  // [0] a wait gave up; [1] wait limit in microseconds (0: default)
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

// Longest-first order of the grid: the clusters of one launch start in grid
// order as SMs free up, so a long query row that starts late sets the launch's
// length.  Grid row `row` takes the query row with the row-th longest causal
// history (ties: lower row first).  Up to kRankMax rows (and kRankSeqMax
// sequences) every CTA ranks them itself in `scratch` (2 kRankMax + 2 ints,
// shared memory that is free until the selection); longer batches are taken
// last row first, which is longest first within a causal prefill.  Returns
// the query row and its sequence (*b).  Every thread of the CTA calls this
// (it has block barriers); row < a.T.
constexpr int kRankMax = 256, kRankSeqMax = 1024;
static_assert(sizeof(SelectSmem) >= (2 * kRankMax + 2) * sizeof(int), "ranking scratch fits the selection block");
template <int kT>
__device__ int ordered_query(const IndexerArgs &a, int row, int *scratch, int *b) {
    if (a.grid_order) {
        *b = find_seq(a.cu_q, a.B, row);
        return row;
    }
    if (a.T > kRankMax || a.B > kRankSeqMax) {
        const int t = a.T - 1 - row;
        *b = find_seq(a.cu_q, a.B, t);
        return t;
    }
    int *pos = scratch, *seq = scratch + kRankMax + 1;
    for (int s = threadIdx.x; s < a.B; s += kT) {
        const int c0 = __ldg(a.cu_q + s), c1 = __ldg(a.cu_q + s + 1), len = __ldg(a.seq_lens + s);
        for (int i = c0; i < c1; ++i) {
            pos[i] = len - (c1 - c0) + (i - c0);  // position of query row i
            seq[i] = s;
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < a.T; i += kT) {
        const int pi = pos[i];
        int rank = 0;
        for (int j = 0; j < a.T; ++j) {
            const int pj = pos[j];
            rank += (pj > pi) || (pj == pi && j < i);
        }
        if (rank == row) {
            pos[kRankMax] = i;
            seq[kRankMax] = seq[i];
        }
    }
    __syncthreads();
    const int t = pos[kRankMax];
    *b = seq[kRankMax];
    __syncthreads();  // the scratch is free again
    return t;
}

template <int G, bool kWriteScores>
__global__ void __launch_bounds__(idx_threads<G>(), 1)
    indexer_topk_bf16_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                             IndexerArgs a) {
    using L = IdxLayout<G>;
    constexpr int kIdxThreads = idx_threads<G>();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int key_cap = a.tiles_cap * kTileM;
    uint8_t *sQ = smem;
    uint8_t *sK = sQ + L::kQBytes;
    uint32_t *sKeys = reinterpret_cast<uint32_t *>(sK + (size_t)a.stages * kTileBytes);
    float *sW = reinterpret_cast<float *>(sKeys + (size_t)G * key_cap);
    uint32_t *sHist0 = reinterpret_cast<uint32_t *>(sW + G * kHI);  // [G][256] top-digit histograms
    int32_t *sRows = reinterpret_cast<int32_t *>(sHist0 + G * kHist);  // [2*tiles_cap] cache row per 64-row box
    SelectSmem *ss = reinterpret_cast<SelectSmem *>(sRows + ((2 * a.tiles_cap + 3) & ~3));
    IdxBars *bars = reinterpret_cast<IdxBars *>(ss + 1);
    static_assert(sizeof(SelectSmem) % 16 == 0, "keep the barrier block 16-byte aligned");

    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int crank = (int)cluster.block_rank();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    grid_dep_wait();  // inputs written by the kernel launched just before are visible

    // ---- which query rows this cluster serves
    int b, t0, gn;
    {
        if (G == 1) {
            if ((int)blockIdx.y >= a.T) return;
            t0 = ordered_query<kIdxThreads>(a, blockIdx.y, reinterpret_cast<int *>(ss), &b);
            gn = 1;
        } else {
            // last (longest, in a causal prefill) groups first
            const int g = a.grid_order ? (int)blockIdx.y : (int)(gridDim.y - 1 - blockIdx.y);
            int acc = 0;
            b = -1;
            for (int s = 0; s < a.B; ++s) {
                int nq = __ldg(a.cu_q + s + 1) - __ldg(a.cu_q + s);
                int ng = (nq + G - 1) / G;
                if (g < acc + ng) {
                    b = s;
                    break;
                }
                acc += ng;
            }
            if (b < 0) return;  // past the last group: the whole cluster leaves together
            t0 = __ldg(a.cu_q + b) + (g - acc) * G;
            gn = min(G, __ldg(a.cu_q + b + 1) - t0);
        }
    }
    const int nq_b = __ldg(a.cu_q + b + 1) - __ldg(a.cu_q + b);
    const int pos_first = __ldg(a.seq_lens + b) - nq_b + (t0 - __ldg(a.cu_q + b));
    const int pos_last = pos_first + gn - 1;   // positions of rows t0 .. t0+gn-1
    const int n_total = pos_last + 1;          // history the group needs
    const int tiles_total = (n_total + kTileM - 1) / kTileM;
    const int tpc = (tiles_total + C - 1) / C;
    const int tile0 = min(tiles_total, crank * tpc);
    int n_tiles = min(tiles_total, tile0 + tpc) - tile0;
    if (n_tiles > a.tiles_cap) {  // a sequence longer than max_pages_per_seq * page_size
        if (threadIdx.x == 0) report_error(a.err, kErrBadLen);
        n_tiles = a.tiles_cap;
    }
    const int32_t *pt_row = a.page_table + (size_t)b * a.max_pages;

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->tfull[i], 1);
            mbar_init(&bars->tempty[i], 4);
            mbar_init(&bars->drain[i], 1);
        }
        mbar_init(&bars->qbar, 1);
        bars->abort[0] = 0;
        bars->abort[1] = wait_limit_us(a.err);
        fence_mbar_init();
    }
    for (int i = threadIdx.x; i < G * kHI; i += kIdxThreads) {
        int gi = i / kHI;
        sW[i] = gi < gn ? __ldg(a.head_w + (size_t)(t0 + gi) * kHI + (i % kHI)) : 0.0f;
    }
    for (int i = threadIdx.x; i < G * kHist; i += kIdxThreads) sHist0[i] = 0u;
    // resolve the physical row of every 64-position box of this CTA's range up
    // front, so that the TMA producer never waits on a page-table load
    for (int j = threadIdx.x; j < 2 * n_tiles; j += kIdxThreads) {
        const int p0 = tile0 * kTileM + j * kBox;
        int row = -1;
        if (p0 <= pos_last) {
            const int page = __ldg(pt_row + p0 / a.page_size);
            if (page < 0 || (int64_t)page >= a.num_pages) report_error(a.err, kErrBadPage);
            else row = page * a.page_size + p0 % a.page_size;
        }
        sRows[j] = row;
    }
    if (warp == 1) tmem_alloc(&bars->tmem_slot, L::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_slot;
    volatile int *abort = bars->abort;
    const int wl = abort[1];  // test wait limit in microseconds (0: the default limit)

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_q);
            mbar_arrive_expect_tx(&bars->qbar, (uint32_t)(gn * 2 * kBoxBytes));
            for (int gi = 0; gi < gn; ++gi) {
                tma_load_2d(sQ + gi * kBoxBytes, &tm_q, &bars->qbar, 0, (t0 + gi) * kHI);
                tma_load_2d(sQ + L::kQRegion + gi * kBoxBytes, &tm_q, &bars->qbar, kBox, (t0 + gi) * kHI);
            }
            int issued = 0;
            for (int i = 0; i < n_tiles; ++i) {
                const int s = i % a.stages;
                if (i >= a.stages && !mbar_wait(&bars->empty[s], ((i / a.stages) & 1) ^ 1, a.err, 0x101, abort, wl))
                    break;
                issued = i + 1;
                uint8_t *dst = sK + (size_t)s * kTileBytes;
                int rows[2];
                uint32_t bytes = 0;
                for (int h = 0; h < 2; ++h) {
                    rows[h] = sRows[2 * i + h];
                    if (rows[h] >= 0) bytes += 2 * kBoxBytes;
                }
                mbar_arrive_expect_tx(&bars->full[s], bytes);
                for (int h = 0; h < 2; ++h) {
                    if (rows[h] < 0) continue;
                    tma_load_2d(dst + h * kBoxBytes, &tm_k, &bars->full[s], 0, rows[h]);
                    tma_load_2d(dst + kRegionBytes + h * kBoxBytes, &tm_k, &bars->full[s], kBox, rows[h]);
                }
            }
            if (*abort) {
                // let copies still in flight land before shared memory is released
                volatile int no_abort[2] = {0, 0};
                mbar_wait(&bars->qbar, 0, nullptr, 0, no_abort);
                for (int i = max(0, issued - a.stages); i < issued; ++i)
                    mbar_wait(&bars->full[i % a.stages], (i / a.stages) & 1, nullptr, 0, no_abort);
            }
        }
    } else if (warp == 1 || warp == kIdxIssuer2) {
        if (lane == 0) {
            // ---------------- tcgen05 issuers: tile i by warp 1 (i even) or kIdxIssuer2 (i odd),
            // into accumulator i & 1; each commits its own MMAs
            const int par = warp == 1 ? 0 : 1;
            constexpr uint32_t idesc = idesc_bf16_f32(kTileM, L::kN);
            bool ok = mbar_wait(&bars->qbar, 0, a.err, 0x201, abort, wl);
            const uint32_t q_base = smem_u32(sQ);
            for (int i = par; ok && i < n_tiles; i += 2) {
                const int s = i % a.stages, buf = par;
                if (!mbar_wait(&bars->full[s], (i / a.stages) & 1, a.err, 0x202, abort, wl)) break;
                if (i >= 2 && !mbar_wait(&bars->tempty[buf], ((i >> 1) & 1) ^ 1, a.err, 0x203, abort, wl)) break;
                tc_fence_after();
                const uint32_t k_base = smem_u32(sK + (size_t)s * kTileBytes);
                const uint32_t d = tmem + (uint32_t)(buf * L::kN);
#pragma unroll
                for (int kk = 0; kk < kDI / 16; ++kk) {
                    const uint32_t off = (uint32_t)((kk & 3) * 32);
                    const uint64_t adesc = sdesc_kmajor_sw128(k_base + (kk >> 2) * kRegionBytes + off);
                    const uint64_t bdesc = sdesc_kmajor_sw128(q_base + (kk >> 2) * L::kQRegion + off);
                    mma_bf16_ss(d, adesc, bdesc, idesc, kk > 0 ? 1u : 0u);
                }
                mma_commit(&bars->empty[s]);
                mma_commit(&bars->tfull[buf]);
            }
            if (*abort) {
                // wait for every issued MMA before TMEM is released
                volatile int no_abort[2] = {0, 0};
                mma_commit(&bars->drain[par]);
                mbar_wait(&bars->drain[par], 0, nullptr, 0, no_abort);
            }
        }
    } else if (warp < 6) {
        // ---------------- epilogue: warps 2..5, thread = position row
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        for (int i = 0; i < n_tiles; ++i) {
            const int buf = i & 1;
            const bool ok = mbar_wait(&bars->tfull[buf], (i >> 1) & 1, a.err, 0x301, abort, wl);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            const int l = i * kTileM + row;          // local key slot
            const int pos = (tile0 + i) * kTileM + row;
#pragma unroll
            for (int gi = 0; gi < G; ++gi) {
                const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(buf * L::kN + gi * kHI);
                uint32_t r0[32], r1[32];
                tmem_ld32(taddr, r0);
                tmem_ld32(taddr + 32, r1);
                tmem_wait_ld();
                const float *w = sW + gi * kHI;
                float acc = 0.0f;
#pragma unroll
                for (int j = 0; j < 32; ++j) acc = fmaf(w[j], fmaxf(__uint_as_float(r0[j]), 0.0f), acc);
#pragma unroll
                for (int j = 0; j < 32; ++j) acc = fmaf(w[32 + j], fmaxf(__uint_as_float(r1[j]), 0.0f), acc);
                const bool valid = gi < gn && pos <= pos_first + gi;
                const uint32_t key = valid ? score_key(acc) : 0u;
                sKeys[(size_t)gi * key_cap + l] = key;
                if (valid) red_shared_add(smem_u32(&sHist0[gi * kHist + (key >> 24)]), 1u);
                if (kWriteScores && valid && pos < a.ld_scores) a.scores[(size_t)(t0 + gi) * a.ld_scores + pos] = acc;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->tempty[buf]);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, L::kTmemCols);
    if (threadIdx.x == 0) grid_dep_launch();  // scoring is done: the next kernel may begin launching
    // A CTA that gave up on a wait (its keys are then incomplete; the error is
    // recorded) still runs the selection: every CTA of the cluster must pass
    // the same sequence of cluster barriers, which depends only on
    // cluster-wide totals.

    // ---------------- selection, one query row at a time
    for (int gi = 0; gi < G; ++gi) {
        if (gi >= gn) {
            cluster.sync();
            continue;
        }
        const int n_valid = pos_first + gi + 1;
        int32_t *out = a.indices + (size_t)(t0 + gi) * a.K;
        cluster_topk<kIdxThreads>(sKeys + (size_t)gi * key_cap, n_tiles * kTileM, tile0 * kTileM, n_valid, a.K, out,
                               *ss, sHist0 + gi * kHist);
    }
}

// ---------------------------------------------------------------------------
// Flat variant (bf16): the 128-position tiles of all query rows, row after
// row, are split evenly over one CTA per SM.  A cluster grid covers the SMs
// only where the rows times the cluster size fit them (32 rows on clusters of
// four take 128 of 152 SMs; 160 rows on one-CTA clusters need a second wave),
// and its rows reach their selection together while memory idles; here every
// SM streams the same share of the index-key cache whatever the rows'
// lengths.  Each CTA writes the keys of its positions (the order-preserving
// form of the scores) to a workspace buffer and adds its counts of their top
// 11 bits to the row's histogram there, then adds its number of the row's
// tiles to the row's counter.  The CTA whose addition completes a row selects
// that row's Top-K after its own scoring: one bulk copy stages the row's keys
// in its shared memory (the query slots and the tile ring are free by then)
// and the whole CTA runs a radix select over them.  Warps: 0 TMA, 1 MMA, 2..5
// epilogue, as in the cluster kernel, and all eight in the selection; the
// query rows' Q tiles come through two slots.
constexpr int kFlatThreads = 256;
constexpr int kFlatWarps = kFlatThreads / 32;
constexpr int kFlatRowsMax = 512;           // query rows of one launch (row tables in shared memory)
constexpr int kFlatQSlot = kHI * kDI * 2;   // 16 KB: both 64-column halves of one query row
constexpr int kFlatBarEpi = 1;              // named barrier of the four epilogue warps
constexpr int kFlatCandMax = 256;           // threshold-bucket keys the exact ranking takes
constexpr int kFlatTopBits = 11;            // top digit counted while scoring
constexpr int kFlatHist = 1 << kFlatTopBits;

struct __align__(16) FlatBars {
    uint64_t drain;
    uint64_t full[8], empty[8];
    uint64_t tfull[2], tempty[2];
    uint64_t qfull[2], qempty[2];
    uint64_t staged;  // a selected row's keys have landed in shared memory
    uint32_t tmem_slot;
    int abort[2];     // [0] a wait gave up; [1] wait limit in microseconds (0: default)
    int n_sel;        // rows this CTA selects
    int first_row;
    int32_t scan[16];
};

// Scratch of the one-CTA selection; it overlays the box-row table, which only
// the TMA producer reads.
constexpr int kFlatSelMax = 49152;          // keys the selection takes (the query slots and a five-tile ring)
struct __align__(16) FlatSel {
    uint32_t hist[2048];                    // counts of the next digit
    uint32_t gt_mask[kFlatSelMax / 32];     // per row of 32 positions: keys above the threshold bucket
    uint32_t eq_mask[kFlatSelMax / 32];     // ... and keys in it
    uint32_t cand_key[kFlatCandMax];
    int32_t cand_pos[kFlatCandMax];
    int32_t wscan[16];
    uint32_t bcast[4];
    uint32_t ncand;
    uint32_t pad_[3];
};

// Byte offsets from the 1024-aligned base of the flat kernel's shared memory.
struct FlatLayout {
    size_t k, w, hist, prefix, len, seq, sel, rows, bars, total;
};
__host__ __device__ inline FlatLayout flat_layout(int stages, int T, int cap_tiles) {
    auto r4 = [](size_t x) { return (x + 3) & ~(size_t)3; };
    FlatLayout L;
    L.k = 2 * (size_t)kFlatQSlot;                // two query slots, then the tile ring
    L.w = L.k + (size_t)stages * kTileBytes;     // [2][64] head weights
    L.hist = L.w + 2 * kHI * 4;                  // [2048] top-digit counts
    L.prefix = L.hist + kFlatHist * 4;           // [T + 1] tiles before each row
    L.len = L.prefix + r4(T + 1) * 4;            // [T] positions each row scores
    L.seq = L.len + r4(T) * 4;                   // [T] sequence of each row
    L.sel = L.seq + r4(T) * 4;                   // [cap] rows this CTA selects
    L.rows = L.sel + r4(cap_tiles) * 4;          // [2 cap] cache row of every 64-position box / FlatSel
    const size_t rows = (size_t)2 * cap_tiles * 4;
    L.bars = L.rows + (rows > sizeof(FlatSel) ? rows : sizeof(FlatSel));
    L.total = L.bars + sizeof(FlatBars);
    return L;
}

// The row that holds flat tile i (i < prefix[T]): the last row starting at or
// before it, which has at least one tile.
__device__ __forceinline__ int flat_row_of(const int32_t *prefix, int T, int i) {
    int lo = 0, hi = T - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= i) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// One radix digit, from the top: the digit whose bucket of the nb-bin
// histogram (nb a multiple of kFlatThreads, at most 2048) at shared address
// hb holds the krem-th largest counted key, and the number of counted keys
// above that bucket.  Thread t sums bins nb-1-per*t down to nb-per*(t+1); an
// exclusive scan over the threads (descending bins) finds the thread whose
// bins hold the krem-th key, and it walks them.  Every thread returns the
// result.  (If the counts add up to fewer than krem, digit 0 with nothing
// above: every thread still takes the same branch.)
__device__ __forceinline__ void flat_find_digit(uint32_t hb, int nb, int krem, FlatSel &fs, uint32_t *digit,
                                                int *above) {
    const int tid = threadIdx.x, per = nb / kFlatThreads;  // 8 or 4 bins
    const int top = nb - 1 - per * tid;
    uint32_t c[8];
    if (per == 8) {
        const uint4 hi = lds128(hb + 4 * (top - 3)), lo = lds128(hb + 4 * (top - 7));
        c[0] = hi.w; c[1] = hi.z; c[2] = hi.y; c[3] = hi.x;
        c[4] = lo.w; c[5] = lo.z; c[6] = lo.y; c[7] = lo.x;
    } else {
        const uint4 hi = lds128(hb + 4 * (top - 3));
        c[0] = hi.w; c[1] = hi.z; c[2] = hi.y; c[3] = hi.x;
        c[4] = c[5] = c[6] = c[7] = 0u;
    }
    const uint32_t part = ((c[0] + c[1]) + (c[2] + c[3])) + ((c[4] + c[5]) + (c[6] + c[7]));
    if (tid == 0) {
        fs.bcast[0] = 0u;
        fs.bcast[1] = 0u;
    }
    const uint32_t excl = (uint32_t)block_exclusive_scan<kFlatThreads>((int)part, fs.wscan, nullptr);
    const uint32_t kr = (uint32_t)krem;
    if (excl < kr && kr <= excl + part) {
        uint32_t ab = excl;
        int i = 0;
        for (; i < per - 1; ++i) {
            if (ab + c[i] >= kr) break;
            ab += c[i];
        }
        fs.bcast[0] = (uint32_t)(top - i);
        fs.bcast[1] = ab;
    }
    __syncthreads();
    *digit = fs.bcast[0];
    *above = (int)fs.bcast[1];
    __syncthreads();  // bcast and the scan scratch are rewritten by the next call
}

// Top-K of one row held in shared memory, by the whole CTA: keys[0..n) (every
// position valid; n <= kFlatSelMax), hist0 (a shared address) = counts of
// their top 11 bits.  Writes min(K, n) positions in ascending order to out,
// then -1 padding.  Radix select from the top: the top 11 bits from hist0,
// then 11 and 10 more, each digit a pass over the keys still in the
// threshold bucket, until that bucket is taken whole, holds few enough keys
// (kFlatCandMax) to rank exactly by (key descending, position ascending), or
// all 32 bits are fixed (equal keys: lowest positions first).  One more pass
// stores, per row of 32 positions, the ballot of its keys above the bucket
// and of its keys in it; the ranked bucket keys are added to the first, and
// each thread then writes the positions of a contiguous run of rows, in
// order, at the slot an exclusive scan of the runs' counts gives it.
// Shared memory is read through shared addresses.
__device__ void flat_cta_topk(uint32_t *keys, int n, uint32_t hist0, int K, int32_t *out, FlatSel &fs) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (n <= K) {
        for (int l = tid; l < K; l += kFlatThreads) out[l] = l < n ? l : -1;
        return;
    }
    const uint32_t kb = smem_u32(keys), hb = smem_u32(fs.hist);
    const int nq = (n + 3) >> 2;  // groups of four keys (the last one may be partial)

    uint32_t digit;
    int above;
    flat_find_digit(hist0, kFlatHist, K, fs, &digit, &above);
    int krem = K - above;
    int shift = 32 - kFlatTopBits;
    uint32_t prefix = digit << shift, mask = ~0u << shift, cnt = lds32(hist0 + 4 * digit);
    while (cnt != (uint32_t)krem && cnt > (uint32_t)kFlatCandMax && shift > 0) {
        const int width = shift > 10 ? 11 : shift, nshift = shift - width;
        const uint32_t dm = (1u << width) - 1u;
        for (int d = tid; d < kFlatHist; d += kFlatThreads) sts32(hb + 4 * d, 0u);
        __syncthreads();
        // four groups of four keys per thread per step, all loaded before any count
        for (int q0 = tid; q0 < nq; q0 += 4 * kFlatThreads) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int q = q0 + u * kFlatThreads;
                v[u] = q < nq ? lds128(kb + 16 * q) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int l = 4 * (q0 + u * kFlatThreads);
                red_shared_add_if(hb + 4 * ((v[u].x >> nshift) & dm), l < n && (v[u].x & mask) == prefix);
                red_shared_add_if(hb + 4 * ((v[u].y >> nshift) & dm), l + 1 < n && (v[u].y & mask) == prefix);
                red_shared_add_if(hb + 4 * ((v[u].z >> nshift) & dm), l + 2 < n && (v[u].z & mask) == prefix);
                red_shared_add_if(hb + 4 * ((v[u].w >> nshift) & dm), l + 3 < n && (v[u].w & mask) == prefix);
            }
        }
        __syncthreads();
        flat_find_digit(hb, kFlatHist >> (11 - width), krem, fs, &digit, &above);
        digit &= dm;
        krem -= above;
        prefix |= digit << nshift;
        mask |= dm << nshift;
        cnt = lds32(hb + 4 * digit);
        shift = nshift;
        __syncthreads();  // everyone has read the histogram before it is cleared
    }
    // 0: the whole bucket is taken; 1: rank the bucket's keys; 2: equal keys
    const int mode = cnt == (uint32_t)krem ? 0 : (cnt <= (uint32_t)kFlatCandMax ? 1 : 2);
    const uint32_t ck = smem_u32(fs.cand_key), cp = smem_u32(fs.cand_pos), nca = smem_u32(&fs.ncand);
    const uint32_t gm = smem_u32(fs.gt_mask), em = smem_u32(fs.eq_mask);
    const int nrows = (n + 31) >> 5;
    if (tid == 0) sts32(nca, 0u);
    __syncthreads();
    // ---- per row of 32 positions: keys above the bucket, keys in it (eight
    // rows per warp per step, all loaded before any ballot)
    for (int j0 = 8 * warp; j0 < nrows; j0 += 8 * kFlatWarps) {
        uint32_t k[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int p = 32 * (j0 + u) + lane;
            k[u] = p < n ? lds32(kb + 4 * p) : 0u;
        }
        uint32_t bg[8], be[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const bool in = 32 * (j0 + u) + lane < n;
            const uint32_t m = k[u] & mask;
            bg[u] = __ballot_sync(0xffffffffu, in && m > prefix);
            be[u] = __ballot_sync(0xffffffffu, in && m == prefix);
        }
        if (lane < 8) {
            // lane u stores row j0 + u (rows past the end are not stored)
            uint32_t g = bg[0], e = be[0];
#pragma unroll
            for (int u = 1; u < 8; ++u) {
                g = lane == u ? bg[u] : g;
                e = lane == u ? be[u] : e;
            }
            if (j0 + lane < nrows) {
                sts32(gm + 4 * (j0 + lane), g);
                sts32(em + 4 * (j0 + lane), e);
            }
        }
    }
    __syncthreads();
    if (mode == 1) {
        // the bucket's keys (few): list them from the masks
        for (int j = tid; j < nrows; j += kFlatThreads) {
            uint32_t e = lds32(em + 4 * j);
            while (e != 0u) {
                const int p = 32 * j + __ffs(e) - 1;
                e &= e - 1u;
                const uint32_t c = atom_shared_add(nca, 1u);
                if (c < (uint32_t)kFlatCandMax) {
                    sts32(ck + 4 * c, lds32(kb + 4 * p));
                    sts32(cp + 4 * c, (uint32_t)p);
                }
            }
        }
        __syncthreads();
        // rank them; the selected ones join their row's mask
        const int nc = min((int)lds32(nca), kFlatCandMax);
        for (int i = tid; i < nc; i += kFlatThreads) {
            const uint32_t ki = lds32(ck + 4 * i);
            const int pi = (int)lds32(cp + 4 * i);
            int r = 0, j = 0;
            for (; j + 4 <= nc; j += 4) {
                uint32_t kj[4];
                int pj[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    kj[u] = lds32(ck + 4 * (j + u));
                    pj[u] = (int)lds32(cp + 4 * (j + u));
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) r += (kj[u] > ki) || (kj[u] == ki && pj[u] < pi);
            }
            for (; j < nc; ++j) {
                const uint32_t kj = lds32(ck + 4 * j);
                r += (kj > ki) || (kj == ki && (int)lds32(cp + 4 * j) < pi);
            }
            if (r < krem) atomicOr(&fs.gt_mask[pi >> 5], 1u << (pi & 31));
        }
        __syncthreads();
    }
    // ---- each thread's run of rows: count, scan, write in order
    const int per = (nrows + kFlatThreads - 1) / kFlatThreads;
    const int j0 = min(nrows, tid * per), j1 = min(nrows, j0 + per);
    int c_sel = 0, c_eq = 0;
    for (int j = j0; j < j1; ++j) {
        const uint32_t g = lds32(gm + 4 * j), e = lds32(em + 4 * j);
        c_sel += __popc(mode == 0 ? (g | e) : g);
        c_eq += __popc(e);
    }
    int eq_rank = 0;
    if (mode == 2) {
        eq_rank = block_exclusive_scan<kFlatThreads>(c_eq, fs.wscan, nullptr);
        c_sel += min(max(krem - eq_rank, 0), c_eq);
    }
    int slot = block_exclusive_scan<kFlatThreads>(c_sel, fs.wscan, nullptr);
    for (int j = j0; j < j1; ++j) {
        uint32_t s = lds32(gm + 4 * j);
        uint32_t e = lds32(em + 4 * j);
        if (mode == 0) s |= e;
        if (mode == 2) {
            // the bucket's keys in position order: the first krem overall are taken
            while (e != 0u && eq_rank < krem) {
                s |= e & (0u - e);
                e &= e - 1u;
                ++eq_rank;
            }
        }
        while (s != 0u) {
            const int b = __ffs(s) - 1;
            if (slot < K) out[slot] = 32 * j + b;
            ++slot;
            s &= s - 1u;
        }
    }
}

__global__ void __launch_bounds__(kFlatThreads, 1)
    indexer_topk_flat_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                             IndexerArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const FlatLayout L = flat_layout(a.stages, a.T, a.flat_cap_tiles);
    uint8_t *sQ = smem;
    uint8_t *sK = smem + L.k;
    float *sW = reinterpret_cast<float *>(smem + L.w);
    uint32_t *sHist = reinterpret_cast<uint32_t *>(smem + L.hist);
    int32_t *sPrefix = reinterpret_cast<int32_t *>(smem + L.prefix);
    int32_t *sLen = reinterpret_cast<int32_t *>(smem + L.len);
    int32_t *sSeq = reinterpret_cast<int32_t *>(smem + L.seq);
    int32_t *sSel = reinterpret_cast<int32_t *>(smem + L.sel);
    int32_t *sRows = reinterpret_cast<int32_t *>(smem + L.rows);
    FlatBars *bars = reinterpret_cast<FlatBars *>(smem + L.bars);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const int max_len = a.max_pages * a.page_size;
    grid_dep_wait();  // inputs written by the kernel launched just before are visible

    // ---- every query row's length and sequence, and the tiles before it
    {
        const int per = (a.T + kFlatThreads - 1) / kFlatThreads;
        const int r0 = min(a.T, tid * per), r1 = min(a.T, r0 + per);
        int sum = 0;
        for (int r = r0; r < r1; ++r) {
            const int b = find_seq(a.cu_q, a.B, r);
            const int c0 = __ldg(a.cu_q + b), nq = __ldg(a.cu_q + b + 1) - c0;
            const int n = __ldg(a.seq_lens + b) - nq + (r - c0) + 1;  // causal history of row r
            if (n > max_len && blockIdx.x == 0) report_error(a.err, kErrBadLen);
            const int nc = max(0, min(n, max_len));
            sLen[r] = nc;
            sSeq[r] = b;
            sum += (nc + kTileM - 1) / kTileM;
        }
        int total = 0;
        int before = block_exclusive_scan<kFlatThreads>(sum, bars->scan, &total);
        for (int r = r0; r < r1; ++r) {
            sPrefix[r] = before;
            before += (sLen[r] + kTileM - 1) / kTileM;
        }
        if (tid == 0) sPrefix[a.T] = total;
    }
    __syncthreads();
    const int W = sPrefix[a.T], P = (int)gridDim.x, p = (int)blockIdx.x;
    const int s0 = (int)((long long)p * W / P);
    const int n_loc = min((int)((long long)(p + 1) * W / P) - s0, a.flat_cap_tiles);
    const int s1 = s0 + n_loc;
    // rows without a position (a sequence shorter than its query rows) select nothing
    for (int r = p; r < a.T; r += P)
        if (sPrefix[r + 1] == sPrefix[r])
            for (int i = tid; i < a.K; i += kFlatThreads) a.indices[(size_t)r * a.K + i] = -1;
    if (n_loc <= 0) return;  // the whole CTA leaves: it holds no tile and no row

    if (tid == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->tfull[i], 1);
            mbar_init(&bars->tempty[i], 4);
            mbar_init(&bars->qfull[i], 1);
            mbar_init(&bars->qempty[i], 1);
        }
        mbar_init(&bars->staged, 1);
        mbar_init(&bars->drain, 1);
        bars->abort[0] = 0;
        bars->abort[1] = wait_limit_us(a.err);
        bars->n_sel = 0;
        bars->first_row = flat_row_of(sPrefix, a.T, s0);
        fence_mbar_init();
    }
    for (int h = tid; h < kFlatHist; h += kFlatThreads) sHist[h] = 0u;
    // the physical row of every 64-position box of this CTA's tiles, up front
    for (int j = tid; j < 2 * n_loc; j += kFlatThreads) {
        const int i = s0 + (j >> 1);
        const int r = flat_row_of(sPrefix, a.T, i);
        const int p0 = (i - sPrefix[r]) * kTileM + (j & 1) * kBox;
        int row = -1;
        if (p0 < sLen[r]) {
            const int page = __ldg(a.page_table + (size_t)sSeq[r] * a.max_pages + p0 / a.page_size);
            if (page < 0 || (int64_t)page >= a.num_pages) report_error(a.err, kErrBadPage);
            else row = page * a.page_size + p0 % a.page_size;
        }
        sRows[j] = row;
    }
    if (warp == 1) tmem_alloc(&bars->tmem_slot, 128);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_slot;
    volatile int *abort = bars->abort;
    const int wl = abort[1];  // test wait limit in microseconds (0: the default limit)
    const int first_row = bars->first_row;

    // Every role walks the CTA's tiles in order; a tile at or past row_end
    // starts this CTA's next row (k counts them).
    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_q);
            int r = first_row - 1, k = -1, row_end = s0, issued = 0, q_issued = 0;
            for (int li = 0; li < n_loc; ++li) {
                const int i = s0 + li;
                if (i >= row_end) {
                    do ++r;
                    while (sPrefix[r + 1] <= i);
                    row_end = sPrefix[r + 1];
                    ++k;
                    const int slot = k & 1;
                    if (k >= 2 && !mbar_wait(&bars->qempty[slot], ((k - 2) >> 1) & 1, a.err, 0x121, abort, wl)) break;
                    mbar_arrive_expect_tx(&bars->qfull[slot], 2 * kBoxBytes);
                    tma_load_2d(sQ + slot * kFlatQSlot, &tm_q, &bars->qfull[slot], 0, r * kHI);
                    tma_load_2d(sQ + slot * kFlatQSlot + kBoxBytes, &tm_q, &bars->qfull[slot], kBox, r * kHI);
                    q_issued = k + 1;
                }
                const int s = li % a.stages;
                if (li >= a.stages && !mbar_wait(&bars->empty[s], ((li / a.stages) & 1) ^ 1, a.err, 0x122, abort, wl))
                    break;
                issued = li + 1;
                uint8_t *dst = sK + (size_t)s * kTileBytes;
                int rows[2];
                uint32_t bytes = 0;
                for (int h = 0; h < 2; ++h) {
                    rows[h] = sRows[2 * li + h];
                    if (rows[h] >= 0) bytes += 2 * kBoxBytes;
                }
                mbar_arrive_expect_tx(&bars->full[s], bytes);
                for (int h = 0; h < 2; ++h) {
                    if (rows[h] < 0) continue;
                    tma_load_2d(dst + h * kBoxBytes, &tm_k, &bars->full[s], 0, rows[h]);
                    tma_load_2d(dst + kRegionBytes + h * kBoxBytes, &tm_k, &bars->full[s], kBox, rows[h]);
                }
            }
            if (*abort) {
                // let copies still in flight land before shared memory is reused or released
                volatile int no_abort[2] = {0, 0};
                for (int kk = max(0, q_issued - 2); kk < q_issued; ++kk)
                    mbar_wait(&bars->qfull[kk & 1], (kk >> 1) & 1, nullptr, 0, no_abort);
                for (int li = max(0, issued - a.stages); li < issued; ++li)
                    mbar_wait(&bars->full[li % a.stages], (li / a.stages) & 1, nullptr, 0, no_abort);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- tcgen05 issuer: D[128 positions x 64 heads] per tile
            constexpr uint32_t idesc = idesc_bf16_f32(kTileM, kHI);
            int r = first_row - 1, k = -1, row_end = s0;
            for (int li = 0; li < n_loc; ++li) {
                const int i = s0 + li;
                if (i >= row_end) {
                    do ++r;
                    while (sPrefix[r + 1] <= i);
                    row_end = sPrefix[r + 1];
                    ++k;
                    if (!mbar_wait(&bars->qfull[k & 1], (k >> 1) & 1, a.err, 0x221, abort, wl)) break;
                }
                const int s = li % a.stages, buf = li & 1;
                if (!mbar_wait(&bars->full[s], (li / a.stages) & 1, a.err, 0x222, abort, wl)) break;
                if (li >= 2 && !mbar_wait(&bars->tempty[buf], ((li >> 1) & 1) ^ 1, a.err, 0x223, abort, wl)) break;
                tc_fence_after();
                const uint32_t k_base = smem_u32(sK + (size_t)s * kTileBytes);
                const uint32_t q_base = smem_u32(sQ + (k & 1) * kFlatQSlot);
                const uint32_t d = tmem + (uint32_t)(buf * kHI);
#pragma unroll
                for (int kk = 0; kk < kDI / 16; ++kk) {
                    const uint32_t off = (uint32_t)((kk & 3) * 32);
                    const uint64_t adesc = sdesc_kmajor_sw128(k_base + (kk >> 2) * kRegionBytes + off);
                    const uint64_t bdesc = sdesc_kmajor_sw128(q_base + (kk >> 2) * kBoxBytes + off);
                    mma_bf16_ss(d, adesc, bdesc, idesc, kk > 0 ? 1u : 0u);
                }
                mma_commit(&bars->empty[s]);
                mma_commit(&bars->tfull[buf]);
                if (i + 1 == row_end || li + 1 == n_loc) mma_commit(&bars->qempty[k & 1]);
            }
            if (*abort) {
                // wait for every issued MMA before TMEM is released
                volatile int no_abort[2] = {0, 0};
                mma_commit(&bars->drain);
                mbar_wait(&bars->drain, 0, nullptr, 0, no_abort);
            }
        }
    } else if (warp < 6) {
        // ---------------- epilogue: warps 2..5, thread = position row of the tile
        // (warps 6 and 7 wait for the selection)
        const int quad = warp & 3, te = tid - 64;
        const int row_t = quad * 32 + lane;
        int r = first_row - 1, k = -1, row_end = s0, n = 0;
        bool ok = true;  // equal across each warp; equal across the four warps at row ends
        for (int li = 0; li < n_loc; ++li) {
            const int i = s0 + li;
            if (i >= row_end) {
                do ++r;
                while (sPrefix[r + 1] <= i);
                row_end = sPrefix[r + 1];
                ++k;
                n = sLen[r];
                if (te < kHI) sW[(k & 1) * kHI + te] = __ldg(a.head_w + (size_t)r * kHI + te);
                bar_sync(kFlatBarEpi, 128);
            }
            const int buf = li & 1;
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->tfull[buf], (li >> 1) & 1, a.err, 0x321, abort, wl));
            if (ok) {
                tc_fence_after();
                const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(buf * kHI);
                uint32_t r0[32], r1[32];
                tmem_ld32(taddr, r0);
                tmem_ld32(taddr + 32, r1);
                tmem_wait_ld();
                const float *w = sW + (k & 1) * kHI;
                float acc = 0.0f;
#pragma unroll
                for (int j = 0; j < 32; ++j) acc = fmaf(w[j], fmaxf(__uint_as_float(r0[j]), 0.0f), acc);
#pragma unroll
                for (int j = 0; j < 32; ++j) acc = fmaf(w[32 + j], fmaxf(__uint_as_float(r1[j]), 0.0f), acc);
                const int pos = (i - sPrefix[r]) * kTileM + row_t;
                if (pos < n) {
                    const uint32_t key = score_key(acc);
                    a.flat_keys[(size_t)r * a.ld_flat + pos] = key;
                    red_shared_add(smem_u32(&sHist[key >> (32 - kFlatTopBits)]), 1u);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->tempty[buf]);
            }
            if (i + 1 == row_end || li + 1 == n_loc) {
                // this CTA's tiles of row r are scored: publish its counts, then its tiles
                ok = bar_and(kFlatBarEpi, 128, ok);
                if (ok) {
                    for (int h = te; h < kFlatHist; h += 128) {
                        const uint32_t v = sHist[h];
                        if (v) atomicAdd(a.flat_hist + (size_t)r * kFlatHist + h, v);
                        sHist[h] = 0u;
                    }
                    __threadfence();
                }
                bar_sync(kFlatBarEpi, 128);
                if (ok && te == 0) {
                    const int mine = min(s1, row_end) - max(s0, sPrefix[r]);
                    const int old = atomicAdd(a.flat_cnt + r, mine);
                    if (old + mine == row_end - sPrefix[r]) {
                        __threadfence();
                        sSel[bars->n_sel++] = r;
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 128);
    if (tid == 0) grid_dep_launch();  // scoring is done: the next kernel may begin launching

    // ---------------- selection of the rows this CTA completed
    uint32_t *stage = reinterpret_cast<uint32_t *>(smem);  // query slots and tile ring, free now
    FlatSel &fs = *reinterpret_cast<FlatSel *>(sRows);
    const int n_sel = bars->n_sel;
    for (int si = 0; si < n_sel; ++si) {
        const int r = sSel[si];
        const int n = sLen[r];
        if (tid == 0) {
            // the other CTAs' key stores (ordered before their counter
            // additions) and this CTA's earlier use of the buffer come before
            // the bulk copy
            fence_proxy_async_global();
            fence_proxy_async_smem();
            const uint32_t bytes = (uint32_t)((n + 3) & ~3) * 4u;
            mbar_arrive_expect_tx(&bars->staged, bytes);
            const uint8_t *src = reinterpret_cast<const uint8_t *>(a.flat_keys + (size_t)r * a.ld_flat);
            for (uint32_t o = 0; o < bytes; o += 32768u)
                bulk_load(reinterpret_cast<uint8_t *>(stage) + o, src + o, min(32768u, bytes - o), &bars->staged);
        }
        for (int h = tid; h < kFlatHist; h += kFlatThreads) sHist[h] = __ldcg(a.flat_hist + (size_t)r * kFlatHist + h);
        const bool landed = mbar_wait(&bars->staged, si & 1, a.err, 0x421, abort, wl);
        if (!__syncthreads_and(landed)) {
            // the row stays unselected (the error is recorded); the copy lands before the CTA leaves
            volatile int no_abort[2] = {0, 0};
            if (tid == 0) mbar_wait(&bars->staged, si & 1, nullptr, 0, no_abort);
            break;
        }
        flat_cta_topk(stage, n, smem_u32(sHist), a.K, a.indices + (size_t)r * a.K, fs);
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// MXFP8 variant: q_idx and the index-key cache are E4M3 with one E8M0 scale per
// 32 consecutive values ("Day-0 Inference Adaptation and Optimization for
// Hybrid Attention Architectures", §4 Optimization 2).  A 128-byte K-major row
// holds all 128 dims of a position, and one block-scaled MMA
// (kind::mxf8f6f4, K = 32) covers exactly one scale group: the tensor core
// multiplies each group's products by 2^(scale_q + scale_k) itself, so the
// four MMAs of a tile accumulate into one accumulator
//     score = sum_j w_j ReLU( sum_g 2^(sq_jg + sk_g) * (q_jg . k_g) )
// and the epilogue is the bf16 kernel's ReLU and head weighting.  The scales
// go to TMEM: the query's once, each key tile's (128 positions x 4 groups)
// into one of two scale buffers, written by four warps (one per lane
// quadrant) ahead of the MMA.
// One cluster serves G query rows of one sequence (G = 1 for decode, 2 in a
// prefill, where consecutive rows read the same history): the G rows' queries
// are stacked in the MMA's N dimension (64 G), so each key tile is read once
// for all of them.  Warps: 0 and 11 TMA, 1 and 10 MMA (even and odd tiles
// each: one thread's waits, issues and commits for a tile take longer than
// the copy engine and the tensor core need for it; with an even ring depth a
// stage belongs to one producer and one issuer), 2..5 epilogue (one per
// TMEM lane quadrant, thread = position, all 64 heads of every row), 6..9
// block scales into TMEM.
constexpr int kF8Threads = 384;
constexpr int kF8Issuer2 = 10;
constexpr int kF8Producer2 = 11;
constexpr int kF8TileBytes = kTileM * kDI;      // 16 KB of E4M3 keys per tile
constexpr int kF8BoxBytes = kBox * kDI;         // 8 KB per 64-row box

struct __align__(16) F8Bars {
    uint64_t full[8];
    uint64_t empty[8];
    uint64_t tfull[4];    // accumulator i % bufs holds tile i
    uint64_t tempty[4];
    uint64_t sf_full[4];  // tile i's key scales are in TMEM scale buffer i % bufs
    uint64_t qbar;
    uint64_t drain[2];  // one per issuing thread
    uint32_t tmem_slot;
    int abort[2];  // [0] a wait gave up; [1] wait limit in microseconds (0: default)
};
// TMEM columns of the MXFP8 kernel: kBufs accumulators of 64 G columns, the
// queries' scales (4 columns: row r of the stacked queries in lane r % 32,
// column r / 32), kBufs key scale buffers (4-aligned).  Several of each keep
// the scale writes (which share TMEM with the running MMA) a few tiles ahead.
template <int G>
struct F8Layout {
    static constexpr int kN = G * kHI;                   // MMA N: the stacked query rows' heads
    static constexpr int kBufs = G == 1 ? 4 : (G == 2 ? 3 : 2);
    static constexpr int kSfQCols = kN <= 128 ? 4 : 8;   // query scale columns (N / 32, 4-aligned)
    static constexpr uint32_t kAccCols = kN, kSfQ = kBufs * kN, kSfK = kSfQ + kSfQCols;
    static_assert(kSfK + 4 * kBufs <= 512, "TMEM");
    static_assert(kN <= 256, "the query scales fill eight TMEM columns at most");
};

// One position's score for one query row from its 64 head logits (TMEM
// accumulator columns): sum_h w_h ReLU(logit_h), as four independent pairs of
// partial sums (heads 8m + 0,1 / 2,3 / 4,5 / 6,7) so that the additions do not
// wait on one another.
__device__ __forceinline__ float f8_row_score(const uint32_t (&r)[64], const float *w_row) {
    float2 p[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f),
                   make_float2(0.0f, 0.0f)};
    const float4 *w4 = reinterpret_cast<const float4 *>(w_row);
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const float4 w = w4[k];
        const int c = 2 * (k & 1);
        p[c] = __ffma2_rn(make_float2(w.x, w.y),
                          make_float2(fmaxf(__uint_as_float(r[4 * k]), 0.0f), fmaxf(__uint_as_float(r[4 * k + 1]), 0.0f)),
                          p[c]);
        p[c + 1] = __ffma2_rn(make_float2(w.z, w.w),
                              make_float2(fmaxf(__uint_as_float(r[4 * k + 2]), 0.0f),
                                          fmaxf(__uint_as_float(r[4 * k + 3]), 0.0f)),
                              p[c + 1]);
    }
    return ((p[0].x + p[1].x) + (p[2].x + p[3].x)) + ((p[0].y + p[1].y) + (p[2].y + p[3].y));
}

// kQuantQ: the query arrives in bf16 and is quantised here, by the scale
// warps, with the standalone quantiser's rule (mxfp8.cuh): codes into the
// query tile in the layout TMA would have written, scales into TMEM.  One
// launch fewer per step than quantising it beforehand.
template <int G, bool kWriteScores, bool kQuantQ>
__global__ void __launch_bounds__(kF8Threads, 1)
    indexer_topk_mxfp8_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                              IndexerArgs a) {
    using L = F8Layout<G>;
    constexpr int kBufs = L::kBufs;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int key_cap = a.tiles_cap * kTileM;
    uint8_t *sQ = smem;                                   // G x 64 heads x 128 B
    uint8_t *sK = sQ + G * kHI * kDI;                     // stages x 16 KB
    uint32_t *sKeys = reinterpret_cast<uint32_t *>(sK + (size_t)a.stages * kF8TileBytes);
    float *sW = reinterpret_cast<float *>(sKeys + (size_t)G * key_cap);
    uint32_t *sHist0 = reinterpret_cast<uint32_t *>(sW + G * kHI);
    int32_t *sRows = reinterpret_cast<int32_t *>(sHist0 + G * kHist);
    SelectSmem *ss = reinterpret_cast<SelectSmem *>(sRows + ((2 * a.tiles_cap + 3) & ~3));
    F8Bars *bars = reinterpret_cast<F8Bars *>(ss + 1);

    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int crank = (int)cluster.block_rank();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    grid_dep_wait();  // inputs written by the kernel launched just before are visible
    // ---- which query rows this cluster serves
    int b, t0, gn;
    if (G == 1) {
        if ((int)blockIdx.y >= a.T) return;
        t0 = ordered_query<kF8Threads>(a, blockIdx.y, reinterpret_cast<int *>(ss), &b);
        gn = 1;
    } else {
        // last (longest, in a causal prefill) groups first
        const int g = a.grid_order ? (int)blockIdx.y : (int)(gridDim.y - 1 - blockIdx.y);
        int acc = 0;
        b = -1;
        for (int s = 0; s < a.B; ++s) {
            const int ng = (__ldg(a.cu_q + s + 1) - __ldg(a.cu_q + s) + G - 1) / G;
            if (g < acc + ng) {
                b = s;
                break;
            }
            acc += ng;
        }
        if (b < 0) return;  // past the last group: the whole cluster leaves together
        t0 = __ldg(a.cu_q + b) + (g - acc) * G;
        gn = min(G, __ldg(a.cu_q + b + 1) - t0);
    }
    const int nq_b = __ldg(a.cu_q + b + 1) - __ldg(a.cu_q + b);
    const int pos_first = __ldg(a.seq_lens + b) - nq_b + (t0 - __ldg(a.cu_q + b));
    const int pos_last = pos_first + gn - 1;   // positions of rows t0 .. t0+gn-1
    const int n_total = pos_last + 1;          // history the group needs
    const int tiles_total = (n_total + kTileM - 1) / kTileM;
    const int tpc = (tiles_total + C - 1) / C;
    const int tile0 = min(tiles_total, crank * tpc);
    int n_tiles = min(tiles_total, tile0 + tpc) - tile0;
    if (n_tiles > a.tiles_cap) {
        if (threadIdx.x == 0) report_error(a.err, kErrBadLen);
        n_tiles = a.tiles_cap;
    }
    const int32_t *pt_row = a.page_table + (size_t)b * a.max_pages;

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        for (int i = 0; i < kBufs; ++i) {
            mbar_init(&bars->tfull[i], 1);
            mbar_init(&bars->tempty[i], 4);
            mbar_init(&bars->sf_full[i], 4);
        }
        mbar_init(&bars->qbar, 1);
        mbar_init(&bars->drain[0], 1);
        mbar_init(&bars->drain[1], 1);
        bars->abort[0] = 0;
        bars->abort[1] = wait_limit_us(a.err);
        fence_mbar_init();
    }
    for (int i = threadIdx.x; i < G * kHI; i += kF8Threads)
        sW[i] = i / kHI < gn ? __ldg(a.head_w + (size_t)t0 * kHI + i) : 0.0f;
    for (int i = threadIdx.x; i < G * kHist; i += kF8Threads) sHist0[i] = 0u;
    if constexpr (!kQuantQ && G > 1) {
        // query rows past the group's last row feed MMA columns nobody reads; keep them finite
        for (int i = gn * kHI * kDI / 16 + threadIdx.x; i < G * kHI * kDI / 16; i += kF8Threads)
            reinterpret_cast<uint4 *>(sQ)[i] = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
    }
    for (int j = threadIdx.x; j < 2 * n_tiles; j += kF8Threads) {
        const int p0 = tile0 * kTileM + j * kBox;
        int row = -1;
        if (p0 <= pos_last) {
            const int page = __ldg(pt_row + p0 / a.page_size);
            if (page < 0 || (int64_t)page >= a.num_pages) report_error(a.err, kErrBadPage);
            else row = page * a.page_size + p0 % a.page_size;
        }
        sRows[j] = row;
    }
    if (warp == 1) tmem_alloc(&bars->tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_slot;
    volatile int *abort = bars->abort;
    const int wl = abort[1];  // test wait limit in microseconds (0: the default limit)

    if (warp == 0 || warp == kF8Producer2) {
        if (lane == 0) {
            // tile i by warp 0 (i even; also the query) or kF8Producer2 (i odd)
            const int par = warp == 0 ? 0 : 1;
            tma_prefetch_desc(&tm_k);
            if constexpr (!kQuantQ) {
                if (par == 0) {
                    tma_prefetch_desc(&tm_q);
                    mbar_arrive_expect_tx(&bars->qbar, (uint32_t)(gn * kHI * kDI));
                    for (int gi = 0; gi < gn; ++gi)
                        tma_load_2d(sQ + gi * kHI * kDI, &tm_q, &bars->qbar, 0, (t0 + gi) * kHI);
                }
            }
            int issued = 0;  // one past this thread's last issued tile
            for (int i = par; i < n_tiles; i += 2) {
                const int s = i % a.stages;
                if (i >= a.stages && !mbar_wait(&bars->empty[s], ((i / a.stages) & 1) ^ 1, a.err, 0x121, abort, wl))
                    break;
                issued = i + 1;
                uint32_t bytes = 0;
                for (int h = 0; h < 2; ++h)
                    if (sRows[2 * i + h] >= 0) bytes += kF8BoxBytes;
                mbar_arrive_expect_tx(&bars->full[s], bytes);
                for (int h = 0; h < 2; ++h) {
                    const int row = sRows[2 * i + h];
                    if (row < 0) continue;
                    tma_load_2d(sK + (size_t)s * kF8TileBytes + h * kF8BoxBytes, &tm_k, &bars->full[s], 0, row);
                }
            }
            if (*abort) {
                // let this thread's copies still in flight land before shared memory is released
                volatile int no_abort[2] = {0, 0};
                if (par == 0) mbar_wait(&bars->qbar, 0, nullptr, 0, no_abort);
                for (int i = max(0, issued - a.stages); i < issued; ++i)
                    if ((i & 1) == par) mbar_wait(&bars->full[i % a.stages], (i / a.stages) & 1, nullptr, 0, no_abort);
            }
        }
    } else if (warp == 1 || warp == kF8Issuer2) {
        if (lane == 0) {
            // tile i by warp 1 (i even) or kF8Issuer2 (i odd); each commits its own MMAs
            const int par = warp == 1 ? 0 : 1;
            bool ok = mbar_wait(&bars->qbar, 0, a.err, 0x221, abort, wl);
            const uint32_t q_base = smem_u32(sQ);
            for (int i = par; ok && i < n_tiles; i += 2) {
                const int s = i % a.stages, buf = i % kBufs;
                const uint32_t round = (uint32_t)(i / kBufs) & 1u;
                if (!mbar_wait(&bars->full[s], (i / a.stages) & 1, a.err, 0x222, abort, wl)) break;
                if (i >= kBufs && !mbar_wait(&bars->tempty[buf], round ^ 1u, a.err, 0x223, abort, wl)) break;
                if (!mbar_wait(&bars->sf_full[buf], round, a.err, 0x224, abort, wl)) break;
                tc_fence_after();
                const uint32_t k_base = smem_u32(sK + (size_t)s * kF8TileBytes);
#pragma unroll
                for (int g = 0; g < 4; ++g)  // one scale group of 32 dims per MMA, scale byte g
                    mma_mxf8_ss(tmem + (uint32_t)(buf * L::kAccCols), sdesc_kmajor_sw128(k_base + g * 32),
                                sdesc_kmajor_sw128(q_base + g * 32), idesc_mxf8_e4m3(kTileM, L::kN, g, g),
                                tmem + L::kSfK + 4u * (uint32_t)buf, tmem + L::kSfQ, g > 0 ? 1u : 0u);
                mma_commit(&bars->empty[s]);
                mma_commit(&bars->tfull[buf]);
            }
            if (*abort) {
                volatile int no_abort[2] = {0, 0};
                mma_commit(&bars->drain[par]);
                mbar_wait(&bars->drain[par], 0, nullptr, 0, no_abort);
            }
        }
    } else if (warp < 6) {
        // epilogue: warp -> TMEM lane quadrant; thread = one position, all 64 heads of every row
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lanes = (uint32_t)(quad * 32) << 16;
        for (int i = 0; i < n_tiles; ++i) {
            const int buf = i % kBufs;
            if (!mbar_wait(&bars->tfull[buf], (uint32_t)(i / kBufs) & 1u, a.err, 0x321, abort, wl)) break;
            tc_fence_after();
            const int pos = (tile0 + i) * kTileM + row;
            const uint32_t acc = tmem + lanes + (uint32_t)(buf * L::kAccCols);
            // the score of row gi at this position: key, top-digit count, (score)
            auto emit = [&](int gi, float sc) {
                const bool valid = gi < gn && pos <= pos_first + gi;
                const uint32_t key = valid ? score_key(sc) : 0u;
                sKeys[(size_t)gi * key_cap + i * kTileM + row] = key;
                if (valid) red_shared_add(smem_u32(&sHist0[gi * kHist + (key >> 24)]), 1u);
                if (kWriteScores && valid && pos < a.ld_scores) a.scores[(size_t)(t0 + gi) * a.ld_scores + pos] = sc;
            };
            if constexpr (G <= 2) {
                uint32_t r[G][64];
#pragma unroll
                for (int gi = 0; gi < G; ++gi) {
                    tmem_ld32(acc + gi * kHI, *reinterpret_cast<uint32_t(*)[32]>(r[gi]));
                    tmem_ld32(acc + gi * kHI + 32, *reinterpret_cast<uint32_t(*)[32]>(r[gi] + 32));
                }
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->tempty[buf]);  // the accumulator is in registers
#pragma unroll
                for (int gi = 0; gi < G; ++gi) emit(gi, f8_row_score(r[gi], sW + gi * kHI));
            } else {
                // three rows: 192 columns do not fit in registers at once; row gi + 1
                // loads while row gi is summed, and the accumulator is handed back
                // once the last row is in registers
                static_assert(G == 3, "three stacked rows");
                uint32_t ra[64], rb[64];
                tmem_ld32(acc, *reinterpret_cast<uint32_t(*)[32]>(ra));
                tmem_ld32(acc + 32, *reinterpret_cast<uint32_t(*)[32]>(ra + 32));
                tmem_wait_ld();
                tmem_ld32(acc + kHI, *reinterpret_cast<uint32_t(*)[32]>(rb));
                tmem_ld32(acc + kHI + 32, *reinterpret_cast<uint32_t(*)[32]>(rb + 32));
                emit(0, f8_row_score(ra, sW));
                tmem_wait_ld();
                tmem_ld32(acc + 2 * kHI, *reinterpret_cast<uint32_t(*)[32]>(ra));
                tmem_ld32(acc + 2 * kHI + 32, *reinterpret_cast<uint32_t(*)[32]>(ra + 32));
                emit(1, f8_row_score(rb, sW + kHI));
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->tempty[buf]);
                emit(2, f8_row_score(ra, sW + 2 * kHI));
            }
        }
    } else {
        // block scales into TMEM, ahead of the MMA: warp -> lane quadrant.
        // Row r's four group scales go to lane r % 32 of every quadrant,
        // column base + r / 32, group g in byte g.
        const int quad = warp & 3;
        const uint32_t lanes = (uint32_t)(quad * 32) << 16;
        // the queries' scales, [row][head][group] (one word per head); the
        // selection block is free scratch until the selection
        uint32_t *sQS = reinterpret_cast<uint32_t *>(ss);
        if constexpr (kQuantQ) {
            // thread i of the four warps: head i / 2 of each row, dims
            // 64 (i % 2) .. +63 (two scale groups).  Codes go to the query
            // tile as a TMA box of 64 rows x 128 bytes with the 128-byte
            // swizzle would place them (16-byte chunk c of row h at h * 128 +
            // ((c ^ (h % 8)) << 4)); rows past the group's last row are zero.
            const int i = (warp - 6) * 32 + lane, h = i >> 1, half = i & 1;
#pragma unroll 1
            for (int gi = 0; gi < G; ++gi) {
                uint8_t *row = sQ + (gi * kHI + h) * 128;
                uint32_t sc = 0u;
                if (gi < gn) {
                    const uint4 *src =
                        reinterpret_cast<const uint4 *>(a.q_bf16 + ((size_t)(t0 + gi) * kHI + h) * kDI + 64 * half);
                    uint4 v[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) v[k] = __ldg(src + k);
#pragma unroll
                    for (int g = 0; g < 2; ++g) {
                        const uint32_t w[16] = {v[4 * g].x,     v[4 * g].y,     v[4 * g].z,     v[4 * g].w,
                                                v[4 * g + 1].x, v[4 * g + 1].y, v[4 * g + 1].z, v[4 * g + 1].w,
                                                v[4 * g + 2].x, v[4 * g + 2].y, v[4 * g + 2].z, v[4 * g + 2].w,
                                                v[4 * g + 3].x, v[4 * g + 3].y, v[4 * g + 3].z, v[4 * g + 3].w};
                        uint32_t out[8];
                        sc |= (uint32_t)mxfp8_block(w, out) << (8 * g);
                        const int c0 = 2 * (2 * half + g);  // first 16-byte chunk of this group in the row
                        *reinterpret_cast<uint4 *>(row + ((c0 ^ (h & 7)) << 4)) = make_uint4(out[0], out[1], out[2], out[3]);
                        *reinterpret_cast<uint4 *>(row + (((c0 + 1) ^ (h & 7)) << 4)) =
                            make_uint4(out[4], out[5], out[6], out[7]);
                    }
                } else {
                    sc = 0x7F7Fu;
#pragma unroll
                    for (int c = 4 * half; c < 4 * half + 4; ++c)
                        *reinterpret_cast<uint4 *>(row + (c << 4)) = make_uint4(0u, 0u, 0u, 0u);
                }
                // groups 2 half, 2 half + 1 of head h: bytes 2 half .. 2 half + 1 of its word
                const uint32_t other = __shfl_xor_sync(0xffffffffu, sc, 1);
                if (half == 0) sQS[gi * kHI + h] = sc | (other << 16);
            }
            fence_proxy_async_smem();  // the codes are read by the tensor cores
            bar_sync(3, 128);          // the four scale warps
            if (threadIdx.x == 6 * 32) mbar_arrive(&bars->qbar);
        }
        if (n_tiles > 0) {
            uint32_t w[L::kSfQCols];  // stacked query row r = gi * 64 + head in lane r % 32, column r / 32
#pragma unroll
            for (int c = 0; c < L::kSfQCols; ++c) {
                const int r = lane + 32 * c, gi = r / kHI, h = r % kHI;
                if (gi >= gn || gi >= G)
                    w[c] = 0x7F7F7F7Fu;
                else if constexpr (kQuantQ)
                    w[c] = sQS[r];
                else
                    w[c] = __ldg(reinterpret_cast<const uint32_t *>(a.q_scale + ((size_t)(t0 + gi) * kHI + h) * 4));
            }
            if constexpr (L::kSfQCols == 4) tmem_st4(tmem + lanes + L::kSfQ, w);
            else tmem_st8(tmem + lanes + L::kSfQ, w);
        }
        // The key scales come straight from the cache with plain loads (a
        // warp's 32 rows are 128 contiguous bytes), issued kBufs tiles
        // ahead: they need only the page rows, not the key tile, and leave the
        // bulk-copy engine to the key tiles.  Rows of a half that is past the
        // sequence get scale 1 (their scores are never used).
        const uint32_t *kscale = reinterpret_cast<const uint32_t *>(a.k_scale);
        auto load_scales = [&](int j, uint32_t (&w)[4]) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int base = sRows[2 * j + (c >> 1)];  // rows 0-63: first box, 64-127: second
                w[c] = base >= 0 ? __ldg(kscale + base + lane + 32 * (c & 1)) : 0x7F7F7F7Fu;
            }
        };
        uint32_t wq[kBufs][4];
#pragma unroll
        for (int u = 0; u < kBufs; ++u)
            if (u < n_tiles) load_scales(u, wq[u]);
        bool sf_ok = true;
        for (int j0 = 0; sf_ok && j0 < n_tiles; j0 += kBufs) {
#pragma unroll
            for (int u = 0; u < kBufs; ++u) {
                const int j = j0 + u;
                if (j >= n_tiles) break;
                // buffer u was last read by the MMA of tile j - kBufs
                if (j >= kBufs &&
                    !mbar_wait(&bars->tfull[u], (uint32_t)((j - kBufs) / kBufs) & 1u, a.err, 0x323, abort, wl)) {
                    sf_ok = false;
                    break;
                }
                tmem_st4(tmem + lanes + L::kSfK + 4u * (uint32_t)u, wq[u]);
                tmem_wait_st();  // (the first time also the queries' scales)
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->sf_full[u]);
                if (j + kBufs < n_tiles) load_scales(j + kBufs, wq[u]);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
    if (threadIdx.x == 0) grid_dep_launch();  // scoring is done: the next kernel may begin launching
    // ---------------- selection, one query row at a time
    for (int gi = 0; gi < G; ++gi) {
        if (gi >= gn) {
            cluster.sync();
            continue;
        }
        int32_t *out = a.indices + (size_t)(t0 + gi) * a.K;
        cluster_topk<kF8Threads>(sKeys + (size_t)gi * key_cap, n_tiles * kTileM, tile0 * kTileM, pos_first + gi + 1,
                                 a.K, out, *ss, sHist0 + gi * kHist);
    }
}

// Top-K of given score rows (test hook and standalone selection).
__global__ void __launch_bounds__(kThreads, 1) topk_from_scores_kernel(TopkArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 15) & ~uintptr_t(15));
    uint32_t *sKeys = reinterpret_cast<uint32_t *>(smem);
    // the selection block needs 16-byte alignment: round the key region up
    SelectSmem *ss = reinterpret_cast<SelectSmem *>(sKeys + ((a.chunk_cap + 3) & ~3));
    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int crank = (int)cluster.block_rank();
    const int r = blockIdx.y;
    if (r >= a.R) return;
    const int n = max(0, min(__ldg(a.lens + r), (int)a.ld));
    const int chunk = (n + C - 1) / C;
    const int p0 = min(n, crank * chunk);
    const int nl = min(n, p0 + chunk) - p0;
    const float *row = a.scores + (size_t)r * a.ld;
    for (int l = threadIdx.x; l < nl; l += kThreads) sKeys[l] = score_key(__ldg(row + p0 + l));
    __syncthreads();
    cluster_topk<kThreads>(sKeys, nl, p0, n, a.K, a.out + (size_t)r * a.K, *ss);
}

}  // namespace

// ------------------------------------------------------------------ host side

size_t indexer_smem_bytes(int G, int stages, int tiles_cap) {
    size_t q = (size_t)G * kHI * kDI * 2;
    size_t k = (size_t)stages * kTileBytes;
    size_t keys = (size_t)G * tiles_cap * kTileM * 4;
    size_t w = (size_t)G * kHI * 4 + (size_t)G * kHist * 4 + (size_t)((2 * tiles_cap + 3) & ~3) * 4;
    return 1024 + q + k + keys + w + sizeof(SelectSmem) + sizeof(IdxBars);
}

size_t indexer_mxfp8_smem_bytes(int G, int stages, int tiles_cap) {
    return 1024 + (size_t)G * kHI * kDI + (size_t)stages * kF8TileBytes + (size_t)G * tiles_cap * kTileM * 4 +
           (size_t)G * (kHI + kHist) * 4 + (size_t)((2 * tiles_cap + 3) & ~3) * 4 + sizeof(SelectSmem) +
           sizeof(F8Bars);
}

template <int G, bool W, bool Q>
static cudaError_t launch_f8(const CUtensorMap &tk, const CUtensorMap &tq, const IndexerArgs &a, int C, int groups,
                             size_t smem, cudaStream_t st) {
    auto kern = indexer_topk_mxfp8_kernel<G, W, Q>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (C > 8) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)C, (unsigned)groups, 1);
    cfg.blockDim = dim3(kF8Threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, tk, tq, a);
}

template <int G>
static cudaError_t launch_f8g(const CUtensorMap &tk, const CUtensorMap &tq, const IndexerArgs &a, int C, int groups,
                              size_t smem, bool write_scores, bool quant_q, cudaStream_t st) {
    if (quant_q)
        return write_scores ? launch_f8<G, true, true>(tk, tq, a, C, groups, smem, st)
                            : launch_f8<G, false, true>(tk, tq, a, C, groups, smem, st);
    return write_scores ? launch_f8<G, true, false>(tk, tq, a, C, groups, smem, st)
                        : launch_f8<G, false, false>(tk, tq, a, C, groups, smem, st);
}

cudaError_t launch_indexer_mxfp8(const CUtensorMap &tm_k, const CUtensorMap &tm_q, const IndexerArgs &a, int G, int C,
                                 int groups, size_t smem, bool write_scores, bool quant_q, cudaStream_t st) {
    // two producers and two issuers on alternate tiles: every stage must belong to one of each
    if (a.stages < 2 || (a.stages & 1) || a.stages > 8) return cudaErrorInvalidValue;
    if (G == 3) return launch_f8g<3>(tm_k, tm_q, a, C, groups, smem, write_scores, quant_q, st);
    if (G == 2) return launch_f8g<2>(tm_k, tm_q, a, C, groups, smem, write_scores, quant_q, st);
    if (G == 1) return launch_f8g<1>(tm_k, tm_q, a, C, groups, smem, write_scores, quant_q, st);
    return cudaErrorInvalidValue;
}

int indexer_mxfp8_max_active_clusters(int G, int C, size_t smem) {
    auto kern = G == 3   ? indexer_topk_mxfp8_kernel<3, false, false>
                : G == 2 ? indexer_topk_mxfp8_kernel<2, false, false>
                         : indexer_topk_mxfp8_kernel<1, false, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 0;
    if (C > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)C, 1, 1);
    cfg.blockDim = dim3(kF8Threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

int indexer_flat_rows_max() { return kFlatRowsMax; }

int indexer_flat_hist_bins() { return kFlatHist; }

int indexer_flat_stage_keys(int stages) {
    const int k = (int)((2 * (size_t)kFlatQSlot + (size_t)stages * kTileBytes) / 4);
    return k < kFlatSelMax ? k : kFlatSelMax;
}

size_t indexer_flat_smem_bytes(int stages, int T, int cap_tiles) {
    return 1024 + flat_layout(stages, T, cap_tiles).total;
}

cudaError_t launch_indexer_flat(const CUtensorMap &tk, const CUtensorMap &tq, const IndexerArgs &a, int ctas,
                                size_t smem, cudaStream_t st) {
    auto kern = indexer_topk_flat_kernel;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas, 1, 1);
    cfg.blockDim = dim3(kFlatThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    // a cluster of one: the selection's barriers then span this CTA alone
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, tk, tq, a);
}

size_t topk_smem_bytes(int chunk_cap) { return 16 + (size_t)((chunk_cap + 3) & ~3) * 4 + sizeof(SelectSmem); }

template <int G, bool W>
static cudaError_t launch_idx(const CUtensorMap &tk, const CUtensorMap &tq, const IndexerArgs &a, int C,
                              int groups, size_t smem, cudaStream_t st) {
    auto kern = indexer_topk_bf16_kernel<G, W>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (C > 8) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)C, (unsigned)groups, 1);
    cfg.blockDim = dim3(idx_threads<G>(), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, tk, tq, a);
}

cudaError_t launch_indexer_bf16(const CUtensorMap &tk, const CUtensorMap &tq, const IndexerArgs &a, int G, int C,
                                int groups, size_t smem, bool write_scores, cudaStream_t st) {
    // two issuing threads on alternate tiles: every stage must belong to one of them
    if (a.stages < 2 || (a.stages & 1) || a.stages > 8) return cudaErrorInvalidValue;
    if (G == 1) return write_scores ? launch_idx<1, true>(tk, tq, a, C, groups, smem, st)
                                    : launch_idx<1, false>(tk, tq, a, C, groups, smem, st);
    if (G == 2) return write_scores ? launch_idx<2, true>(tk, tq, a, C, groups, smem, st)
                                    : launch_idx<2, false>(tk, tq, a, C, groups, smem, st);
    if (G == 4) return write_scores ? launch_idx<4, true>(tk, tq, a, C, groups, smem, st)
                                    : launch_idx<4, false>(tk, tq, a, C, groups, smem, st);
    return cudaErrorInvalidValue;
}

template <int G>
static int max_clusters_g(int C, size_t smem) {
    auto kern = indexer_topk_bf16_kernel<G, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 0;
    if (C > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)C, 1, 1);
    cfg.blockDim = dim3(idx_threads<G>(), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

int indexer_max_active_clusters(int G, int C, size_t smem) {
    if (G == 1) return max_clusters_g<1>(C, smem);
    if (G == 2) return max_clusters_g<2>(C, smem);
    if (G == 4) return max_clusters_g<4>(C, smem);
    return 0;
}

cudaError_t launch_topk_from_scores(const TopkArgs &a, int C, size_t smem, cudaStream_t st) {
    auto kern = topk_from_scores_kernel;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (C > 8) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)C, (unsigned)a.R, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace dsa
