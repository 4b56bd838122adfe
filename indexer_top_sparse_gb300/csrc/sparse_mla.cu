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
// key split, query row); heads are the MMA's N dimension so that the output
// accumulator O^T [512 dims x NH heads] takes 4*NH TMEM columns and the logit
// tile S^T [128 keys x NH heads] another NH.
//   warp 0      gather producer: per tile of 128 selected keys, TMA
//               tile::gather4 copies the 576-wide bf16 rows (resolved through
//               the page table) into nine 64-column regions with the 128-byte
//               swizzle; a region is refilled as soon as the MMAs of the
//               previous tile are done with it.
//   warp 1      tcgen05 issuer: S^T = K_tile * Q^T (K-major operands, 36 steps
//               of K=16), then after the softmax O^T += V^T * P^T with V^T read
//               MN-major from the same smem tile (4 chunks of 128 dims, 8 steps
//               of 16 keys) and P^T K-major.
//   warps 2-9   softmax: thread = key (TMEM lane), each warp half of the heads;
//               per-head max and sum over the 128 keys by a warp transpose
//               reduction plus a 4-way shared-memory combine; exp2 with log2(e)
//               folded into the scale; the reference max moves only when a
//               head's max grows by more than 2^8 (then O^T is rescaled in
//               TMEM); P (bf16) is written over the tile's consumed rope region.
// With several key splits per row, partial (O, max, sum) go to the workspace
// and mla_combine_kernel merges them.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "ptx.cuh"
#include "kernels.h"

namespace dsa {

namespace {

constexpr int kDv = 512;
constexpr int kHG = 64;                      // head-slot stride of the partial layout
constexpr int kKeys = 128;                   // keys per tile (MMA M of S^T)
constexpr int kRegions = 9;                  // 64-dim regions of a 576-wide row
constexpr int kRegionBytes = kKeys * 128;    // 16 KB
constexpr int kTileBytes = kRegions * kRegionBytes;
constexpr int kThreads = 320;
constexpr int kSmThreads = 256;              // softmax warps 2..9
constexpr int kBarSm = 1;                    // named barrier of the softmax warps

template <int NH>
struct MlaLayout {
    static constexpr int kQRegion = NH * 128;
    static constexpr int kQBytes = kRegions * kQRegion;
    static constexpr int kKVOff = kQBytes;
    static constexpr int kPOff = kKVOff + 8 * kRegionBytes;  // the rope region doubles as P
    static constexpr int kPHalf = NH * 128;                    // P^T rows for 64 keys
    static constexpr int kMiscOff = kKVOff + kTileBytes;
    static constexpr int kTmemCols = 5 * NH <= 128 ? 128 : (5 * NH <= 256 ? 256 : 512);
    static_assert(kQBytes % 1024 == 0, "regions must stay 1024-byte aligned");
};

struct __align__(16) MlaBars {
    uint64_t reg_full[kRegions];
    uint64_t reg_empty[kRegions];
    uint64_t s_full, p_full, o_full, q_full, drain;
    uint32_t tmem_slot;
    int abort;
};

struct __align__(16) MlaStats {
    float red[4][kHG];
    float red2[4][kHG];
    float m_ref[kHG];
    float l_run[kHG];
    float alpha[kHG];
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ int find_seq(const int32_t *cu_q, int B, int t) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (__ldg(cu_q + mid) <= t) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

template <int N>
struct Log2 {
    static constexpr int v = N <= 1 ? 0 : 1 + Log2<N / 2>::v;
};
template <>
struct Log2<1> {
    static constexpr int v = 0;
};

// Reduce N per-head values over the 32 lanes of a warp.  Halving exchanges
// leave each lane with one head; the remaining offsets finish the reduction.
// Returns the reduced value; *head receives which of the N heads it is.
template <int N, bool kMax>
__device__ __forceinline__ float warp_reduce_heads(float (&v)[N], int lane, int *head) {
    constexpr int L = Log2<N>::v;
    int h = 0;
#pragma unroll
    for (int s = 0; s < L; ++s) {
        const int o = 16 >> s;
        const int half = N >> (s + 1);
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float keep = up ? v[i + half] : v[i];
            const float send = up ? v[i] : v[i + half];
            const float recv = __shfl_xor_sync(0xffffffffu, send, o);
            v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
        }
        h += up ? half : 0;
    }
#pragma unroll
    for (int o = 16 >> L; o >= 1; o >>= 1) {
        const float r = __shfl_xor_sync(0xffffffffu, v[0], o);
        v[0] = kMax ? fmaxf(v[0], r) : v[0] + r;
    }
    *head = h;
    return v[0];
}

template <int NH>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_mla_tc_kernel(const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_q,
                         MlaArgs a) {
    using L = MlaLayout<NH>;
    constexpr int HW = NH / 2;  // heads per softmax warp
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQ = smem;
    uint8_t *sKV = smem + L::kKVOff;
    uint8_t *sP = smem + L::kPOff;
    MlaBars *bars = reinterpret_cast<MlaBars *>(smem + L::kMiscOff);
    MlaStats *st = reinterpret_cast<MlaStats *>(bars + 1);

    const int hg = blockIdx.x, split = blockIdx.y, t = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int k_begin = split * a.keys_per_split;
    const int k_end = min(a.K, k_begin + a.keys_per_split);
    const int n_tiles = k_end > k_begin ? (k_end - k_begin + kKeys - 1) / kKeys : 0;
    const int b = find_seq(a.cu_q, a.B, t);
    const int pos = __ldg(a.seq_lens + b) - (__ldg(a.cu_q + b + 1) - __ldg(a.cu_q + b)) + (t - __ldg(a.cu_q + b));
    const int32_t *idx_row = a.indices + (size_t)t * a.K;

    if (threadIdx.x == 0) {
        for (int r = 0; r < kRegions; ++r) {
            mbar_init(&bars->reg_full[r], 1);
            mbar_init(&bars->reg_empty[r], 1);
        }
        mbar_init(&bars->s_full, 1);
        mbar_init(&bars->p_full, kSmThreads / 32);
        mbar_init(&bars->o_full, 1);
        mbar_init(&bars->q_full, 1);
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbar_init();
    }
    if (threadIdx.x < NH) {
        st->m_ref[threadIdx.x] = -CUDART_INF_F;
        st->l_run[threadIdx.x] = 0.0f;
    }
    if (warp == 1) tmem_alloc(&bars->tmem_slot, L::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_o = bars->tmem_slot;          // O^T: columns [0, 4*NH)
    const uint32_t tmem_s = tmem_o + 4 * NH;          // S^T: columns [4*NH, 5*NH)
    volatile int *abort = &bars->abort;

    if (warp == 0) {
        // ---------------------------------------------------------------- gather producer
        const int32_t *pt_row = a.page_table + (size_t)b * a.max_pages;
        if (lane == 0) {
            tma_prefetch_desc(&tm_kv);
            tma_prefetch_desc(&tm_q);
            mbar_arrive_expect_tx(&bars->q_full, (uint32_t)(kRegions * L::kQRegion));
            for (int r = 0; r < kRegions; ++r)
                tma_load_2d(sQ + r * L::kQRegion, &tm_q, &bars->q_full, 64 * r, t * a.H + hg * NH);
        }
        int last_tile = -1, last_regions = 0;
        for (int i = 0; i < n_tiles; ++i) {
            int rows[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                rows[j] = 0;  // invalid slots read row 0 and are masked by the softmax
                const int slot = k_begin + i * kKeys + 4 * lane + j;
                if (slot < k_end) {
                    const int idx = __ldg(idx_row + slot);
                    if (idx > pos) {
                        report_error(a.err, kErrBadIndex);
                    } else if (idx >= 0) {
                        const int page = __ldg(pt_row + idx / a.page_size);
                        if (page < 0 || (int64_t)page >= a.num_pages)
                            report_error(a.err, kErrBadPage);
                        else
                            rows[j] = page * a.page_size + idx % a.page_size;
                    }
                }
            }
            bool stop = false;
            for (int r = 0; r < kRegions; ++r) {
                bool ok = true;
                if (i > 0) ok = mbar_wait(&bars->reg_empty[r], (i - 1) & 1, a.err, 0x501, abort);
                if (!__all_sync(0xffffffffu, ok)) {
                    stop = true;
                    break;
                }
                if (lane == 0) mbar_arrive_expect_tx(&bars->reg_full[r], (uint32_t)kRegionBytes);
                __syncwarp();
                tma_gather4(sKV + r * kRegionBytes + lane * 512, &tm_kv, &bars->reg_full[r], 64 * r, rows[0], rows[1],
                            rows[2], rows[3]);
                last_tile = i;
                last_regions = r + 1;
            }
            if (stop) break;
        }
        if (lane == 0 && *abort) {
            // let the copies in flight land before shared memory is released
            volatile int no_abort = 0;
            mbar_wait(&bars->q_full, 0, nullptr, 0, &no_abort);
            for (int r = 0; r < last_regions; ++r)
                mbar_wait(&bars->reg_full[r], last_tile & 1, nullptr, 0, &no_abort);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- tcgen05 issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(kKeys, NH);
            constexpr uint32_t idesc_o = idesc_bf16_f32_amn(128, NH);
            const uint32_t q_base = smem_u32(sQ), kv_base = smem_u32(sKV), p_base = smem_u32(sP);
            bool ok = mbar_wait(&bars->q_full, 0, a.err, 0x502, abort);
            for (int i = 0; ok && i < n_tiles; ++i) {
                // S^T[128 keys x NH] = K_tile[128 x 576] . Q[NH x 576]^T
                for (int r = 0; r < kRegions && ok; ++r) {
                    ok = mbar_wait(&bars->reg_full[r], i & 1, a.err, 0x503, abort);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = sdesc_kmajor_sw128(kv_base + r * kRegionBytes + kk * 32);
                        const uint64_t bd = sdesc_kmajor_sw128(q_base + r * L::kQRegion + kk * 32);
                        mma_bf16_ss(tmem_s, ad, bd, idesc_s, (r | kk) ? 1u : 0u);
                    }
                }
                if (!ok) break;
                mma_commit(&bars->s_full);
                ok = mbar_wait(&bars->p_full, i & 1, a.err, 0x504, abort);
                if (!ok) break;
                tc_fence_after();
                // O^T[512 x NH] += V^T[512 x 128 keys] . P^T[NH x 128 keys]^T, by 128-dim chunks
                for (int c = 0; c < 4; ++c) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint64_t ad =
                            sdesc_mnmajor_sw128(kv_base + 2 * c * kRegionBytes + j * 2048, kRegionBytes, 1024);
                        const uint64_t bd = sdesc_kmajor_sw128(p_base + (j >> 2) * L::kPHalf + (j & 3) * 32);
                        mma_bf16_ss(tmem_o + c * NH, ad, bd, idesc_o, (i > 0 || j > 0) ? 1u : 0u);
                    }
                    mma_commit(&bars->reg_empty[2 * c]);
                    mma_commit(&bars->reg_empty[2 * c + 1]);
                }
                mma_commit(&bars->reg_empty[8]);
            }
            if (ok && n_tiles > 0) mma_commit(&bars->o_full);
            if (*abort) {
                volatile int no_abort = 0;
                mma_commit(&bars->drain);
                mbar_wait(&bars->drain, 0, nullptr, 0, &no_abort);
            }
        }
    } else {
        // ---------------------------------------------------------------- softmax warps
        const int sw = warp - 2, quad = warp & 3, ch = sw >> 2;
        const int key_local = quad * 32 + lane;
        const int tid_s = sw * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        bool ok = true;
        for (int i = 0; i < n_tiles; ++i) {
            const int slot = k_begin + i * kKeys + key_local;
            bool valid = false;
            if (slot < k_end) {
                const int idx = __ldg(idx_row + slot);
                valid = idx >= 0 && idx <= pos;
            }
            ok = mbar_wait(&bars->s_full, i & 1, a.err, 0x505, abort);
            ok = bar_and(kBarSm, kSmThreads, ok);
            if (!ok) break;
            tc_fence_after();
            uint32_t raw[HW];
            tmem_ld<HW>(tmem_s + lane_off + ch * HW, raw);
            tmem_wait_ld();
            float x[HW], y[HW];
#pragma unroll
            for (int j = 0; j < HW; ++j) {
                x[j] = valid ? __uint_as_float(raw[j]) * a.scale_log2 : -CUDART_INF_F;
                y[j] = x[j];
            }
            int hl;
            const float wmax = warp_reduce_heads<HW, true>(y, lane, &hl);
            st->red[quad][ch * HW + hl] = wmax;
            bar_sync(kBarSm, kSmThreads);
            if (tid_s < NH) {
                const int h = tid_s;
                const float mt = fmaxf(fmaxf(st->red[0][h], st->red[1][h]), fmaxf(st->red[2][h], st->red[3][h]));
                const float mo = st->m_ref[h];
                float al = 1.0f;
                if (mt != -CUDART_INF_F && (mo == -CUDART_INF_F || mt > mo + 8.0f)) {
                    al = mo == -CUDART_INF_F ? 1.0f : exp2f(mo - mt);
                    st->m_ref[h] = mt;
                }
                st->alpha[h] = al;
            }
            bar_sync(kBarSm, kSmThreads);
            float p[HW];
            bool rescale = false;
#pragma unroll
            for (int j = 0; j < HW; ++j) {
                const float m = st->m_ref[ch * HW + j];
                p[j] = exp2f(x[j] - (m == -CUDART_INF_F ? 0.0f : m));
                y[j] = p[j];
                rescale |= st->alpha[ch * HW + j] != 1.0f;
            }
            const float wsum = warp_reduce_heads<HW, false>(y, lane, &hl);
            st->red2[quad][ch * HW + hl] = wsum;
            // P^T (bf16), K-major with the 128-byte swizzle: row = head, column = key
            {
                const int sub = key_local >> 6, col = key_local & 63;
                uint8_t *pbase = sP + sub * L::kPHalf + (col & 7) * 2;
                const int chunk = col >> 3;
#pragma unroll
                for (int j = 0; j < HW; ++j) {
                    const int h = ch * HW + j;
                    __nv_bfloat16 v = __float2bfloat16_rn(p[j]);
                    *reinterpret_cast<__nv_bfloat16 *>(pbase + h * 128 + ((chunk ^ (h & 7)) << 4)) = v;
                }
            }
            if (rescale) {
                // the reference max moved: O^T columns of this warp's heads *= alpha
                float al[HW];
#pragma unroll
                for (int j = 0; j < HW; ++j) al[j] = st->alpha[ch * HW + j];
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t o[HW];
                    const uint32_t ta = tmem_o + lane_off + c * NH + ch * HW;
                    tmem_ld<HW>(ta, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < HW; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * al[j]);
                    tmem_st<HW>(ta, o);
                }
                tmem_wait_st();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            bar_sync(kBarSm, kSmThreads);
            if (tid_s < NH) {
                const int h = tid_s;
                st->l_run[h] = st->l_run[h] * st->alpha[h] + (st->red2[0][h] + st->red2[1][h]) +
                               (st->red2[2][h] + st->red2[3][h]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->p_full);
        }

        // ---------------------------------------------------------------- epilogue
        if (ok && n_tiles > 0) ok = mbar_wait(&bars->o_full, 0, a.err, 0x506, abort);
        ok = bar_and(kBarSm, kSmThreads, ok);
        if (ok) {
            tc_fence_after();
            const int groups = gridDim.x;
            const int h_base = hg * NH + ch * HW;
            float inv[HW];
#pragma unroll
            for (int j = 0; j < HW; ++j) {
                const float l = st->l_run[ch * HW + j];
                inv[j] = (a.splits == 1 && l > 0.0f) ? 1.0f / l : (a.splits == 1 ? 0.0f : 1.0f);
            }
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t o[HW];
                if (n_tiles > 0) {
                    tmem_ld<HW>(tmem_o + lane_off + c * NH + ch * HW, o);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int j = 0; j < HW; ++j) o[j] = 0u;
                }
                const int d = c * 128 + quad * 32 + lane;
                if (a.splits == 1) {
#pragma unroll
                    for (int j = 0; j < HW; ++j)
                        a.out[((size_t)t * a.H + h_base + j) * kDv + d] =
                            __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(o[j]) * inv[j]));
                } else {
                    const size_t slot0 = (((size_t)t * groups + hg) * a.splits + split) * kHG + ch * HW;
#pragma unroll
                    for (int j = 0; j < HW; ++j) a.part_o[(slot0 + j) * kDv + d] = __uint_as_float(o[j]);
                }
            }
            if (tid_s < NH) {
                const int h = tid_s;
                const float l = st->l_run[h], m = st->m_ref[h];
                if (a.splits == 1) {
                    if (a.lse)
                        a.lse[(size_t)t * a.H + hg * NH + h] =
                            l > 0.0f ? m * 0.69314718055994531f + logf(l) : -CUDART_INF_F;
                } else {
                    const size_t slot0 = (((size_t)t * groups + hg) * a.splits + split) * kHG + h;
                    a.part_ml[slot0 * 2 + 0] = l > 0.0f ? m : -CUDART_INF_F;
                    a.part_ml[slot0 * 2 + 1] = l;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_o, L::kTmemCols);
}

// Merge split partials: block = (head, head group, query row), 128 threads x 4 dims.
__global__ void __launch_bounds__(128) mla_combine_kernel(MlaArgs a, int NH) {
    const int hl = blockIdx.x, hg = blockIdx.y, t = blockIdx.z;
    if (hl >= NH) return;
    const int h = hg * NH + hl;
    const size_t base = ((size_t)t * gridDim.y + hg) * a.splits;
    float M = -CUDART_INF_F;
    for (int s = 0; s < a.splits; ++s) M = fmaxf(M, a.part_ml[((base + s) * kHG + hl) * 2]);
    const float ref = M == -CUDART_INF_F ? 0.0f : M;
    float Lsum = 0.0f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < a.splits; ++s) {
        const float ms = a.part_ml[((base + s) * kHG + hl) * 2];
        const float ls = a.part_ml[((base + s) * kHG + hl) * 2 + 1];
        const float w = ls > 0.0f ? exp2f(ms - ref) : 0.0f;
        Lsum += ls * w;
        const float4 v = reinterpret_cast<const float4 *>(a.part_o + ((base + s) * kHG + hl) * kDv)[threadIdx.x];
        acc.x += w * v.x;
        acc.y += w * v.y;
        acc.z += w * v.z;
        acc.w += w * v.w;
    }
    const float inv = Lsum > 0.0f ? 1.0f / Lsum : 0.0f;
    uint32_t *o = reinterpret_cast<uint32_t *>(a.out + ((size_t)t * a.H + h) * kDv);
    o[threadIdx.x * 2] = pack_bf16(acc.x * inv, acc.y * inv);
    o[threadIdx.x * 2 + 1] = pack_bf16(acc.z * inv, acc.w * inv);
    if (a.lse && threadIdx.x == 0)
        a.lse[(size_t)t * a.H + h] = Lsum > 0.0f ? ref * 0.69314718055994531f + logf(Lsum) : -CUDART_INF_F;
}

}  // namespace

size_t mla_smem_bytes(int NH) {
    const size_t q = (size_t)kRegions * NH * 128;
    return 1024 + q + kTileBytes + sizeof(MlaBars) + sizeof(MlaStats);
}
int mla_key_tile() { return kKeys; }

template <int NH>
static cudaError_t launch_tc(const CUtensorMap &tkv, const CUtensorMap &tq, const MlaArgs &a, cudaStream_t st) {
    const size_t smem = mla_smem_bytes(NH);
    auto kern = sparse_mla_tc_kernel<NH>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(a.H / NH, a.splits, a.T), kThreads, smem, st>>>(tkv, tq, a);
    return cudaGetLastError();
}

cudaError_t launch_sparse_mla_bf16(const CUtensorMap &tkv, const CUtensorMap &tq, const MlaArgs &a, int NH,
                                   cudaStream_t st) {
    cudaError_t e;
    if (NH == 64) e = launch_tc<64>(tkv, tq, a, st);
    else if (NH == 32) e = launch_tc<32>(tkv, tq, a, st);
    else if (NH == 16) e = launch_tc<16>(tkv, tq, a, st);
    else return cudaErrorInvalidValue;
    if (e != cudaSuccess || a.splits == 1) return e;
    mla_combine_kernel<<<dim3(kHG, a.H / NH, a.T), 128, 0, st>>>(a, NH);
    return cudaGetLastError();
}

}  // namespace dsa
