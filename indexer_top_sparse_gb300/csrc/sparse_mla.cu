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
// Design: CTA = (64-head group, key split, query row).  A producer warp
// gathers the selected 576-wide bf16 rows (1152 B each, one bulk copy per row)
// through the page table into a 4-deep ring of 32-row tiles, padded to a
// 1168-byte row pitch so that ldmatrix is bank-conflict free.  Eight compute
// warps: warp w owns heads 16*(w%4).. and value dims 256*(w/4)..; each
// computes its 16x32 logit tile with mma.sync m16n8k16 (bf16 in, fp32 acc),
// runs the online softmax in registers (exp2 with log2(e) folded into the
// scale) and accumulates P*V for its 256 value dims.  With several key splits
// per row, partial (O, max, sum) go to the workspace and a combine kernel
// merges them.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "ptx.cuh"
#include "kernels.h"

namespace dsa {

namespace {

constexpr int kD = 576;
constexpr int kDv = 512;
constexpr int kRowBytes = kD * 2;            // 1152
constexpr int kPitch = kRowBytes + 16;       // 1168: 4-bank shift per row
constexpr int kHG = 64;                      // heads per CTA
constexpr int kNT = 32;                      // keys per tile
constexpr int kStages = 4;
constexpr int kComputeWarps = 8;
constexpr int kThreads = (kComputeWarps + 1) * 32;
constexpr int kQBytes = kHG * kPitch;
constexpr int kStageBytes = kNT * kPitch;

struct __align__(16) MlaBars {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t qbar;
    int abort;
    int pad;
    uint8_t valid[kStages][kNT];
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
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

__global__ void __launch_bounds__(kThreads, 1) sparse_mla_bf16_kernel(MlaArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    uint8_t *sQ = smem;
    uint8_t *sKV = sQ + kQBytes;
    MlaBars *bars = reinterpret_cast<MlaBars *>(sKV + kStages * kStageBytes);

    const int hg = blockIdx.x, split = blockIdx.y, t = blockIdx.z;
    const int heads_here = min(kHG, a.H - hg * kHG);  // multiple of 16
    const int n_hb = heads_here / 16;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int k_begin = split * a.keys_per_split;
    const int k_end = min(a.K, k_begin + a.keys_per_split);
    const int n_tiles = k_end > k_begin ? (k_end - k_begin + kNT - 1) / kNT : 0;
    const int active_warps = 2 * n_hb;

    // zero the ring once so that rows never loaded read as finite zeros
    for (int i = threadIdx.x; i < kStages * kStageBytes / 16; i += kThreads)
        reinterpret_cast<uint4 *>(sKV)[i] = make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], active_warps);
        }
        mbar_init(&bars->qbar, 1);
        bars->abort = 0;
        fence_mbar_init();
    }
    fence_proxy_async_smem();
    __syncthreads();
    volatile int *abort = &bars->abort;

    if (warp == kComputeWarps) {
        // ---------------- gather producer (whole warp; lane = key slot)
        const int b = find_seq(a.cu_q, a.B, t);
        const int nq = __ldg(a.cu_q + b + 1) - __ldg(a.cu_q + b);
        const int pos = __ldg(a.seq_lens + b) - nq + (t - __ldg(a.cu_q + b));
        const int32_t *pt_row = a.page_table + (size_t)b * a.max_pages;
        const int32_t *idx_row = a.indices + (size_t)t * a.K;
        const uint8_t *qsrc = reinterpret_cast<const uint8_t *>(a.q + ((size_t)t * a.H + hg * kHG) * kD);
        if (lane == 0) mbar_arrive_expect_tx(&bars->qbar, (uint32_t)(heads_here * kRowBytes));
        __syncwarp();
        for (int h = lane; h < heads_here; h += 32)
            bulk_load(sQ + h * kPitch, qsrc + (size_t)h * kRowBytes, kRowBytes, &bars->qbar);
        int issued = 0;
        for (int i = 0; i < n_tiles; ++i) {
            const int s = i % kStages;
            bool ok = true;
            if (i >= kStages) ok = mbar_wait(&bars->empty[s], ((i / kStages) & 1) ^ 1, a.err, 0x401, abort);
            if (!__all_sync(0xffffffffu, ok)) break;
            const int slot = k_begin + i * kNT + lane;
            long long row = -1;
            if (slot < k_end) {
                const int idx = __ldg(idx_row + slot);
                if (idx >= 0) {
                    if (idx > pos) {
                        report_error(a.err, kErrBadIndex);
                    } else {
                        const int page = __ldg(pt_row + idx / a.page_size);
                        if (page < 0 || (int64_t)page >= a.num_pages)
                            report_error(a.err, kErrBadPage);
                        else
                            row = (long long)page * a.page_size + idx % a.page_size;
                    }
                }
            }
            const bool v = row >= 0;
            bars->valid[s][lane] = v ? 1 : 0;
            const unsigned ball = __ballot_sync(0xffffffffu, v);
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(&bars->full[s], (uint32_t)(__popc(ball) * kRowBytes));
            __syncwarp();
            if (v) bulk_load(sKV + s * kStageBytes + lane * kPitch, a.kv + row * kRowBytes, kRowBytes, &bars->full[s]);
            issued = i + 1;
        }
        // keep the CTA alive until the copies it issued have landed, even if
        // the compute warps stopped early
        if (lane == 0) {
            volatile int no_abort = 0;
            mbar_wait(&bars->qbar, 0, nullptr, 0, &no_abort);
            for (int i = max(0, issued - kStages); i < issued; ++i)
                mbar_wait(&bars->full[i % kStages], (i / kStages) & 1, nullptr, 0, &no_abort);
        }
        return;
    }
    const int hb = warp & 3, dh = warp >> 2;
    if (hb >= n_hb) return;

    // ---------------- compute warps
    const int g = lane >> 2, q4 = lane & 3;  // mma fragment coordinates
    float o[32][4];
#pragma unroll
    for (int n = 0; n < 32; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.0f;
    float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.0f, l1 = 0.0f;

    const bool qok = mbar_wait(&bars->qbar, 0, a.err, 0x402, abort);
    const uint32_t q_addr = smem_u32(sQ) + (uint32_t)((hb * 16 + (lane & 15)) * kPitch + (lane >> 4) * 16);
    for (int i = 0; qok && i < n_tiles; ++i) {
        const int s = i % kStages;
        const bool ok = mbar_wait(&bars->full[s], (i / kStages) & 1, a.err, 0x403, abort);
        if (!__all_sync(0xffffffffu, ok)) break;
        const uint32_t kv_base = smem_u32(sKV + s * kStageBytes);

        // S[16 heads x 32 keys] = Q_hb . K^T over 576 dims
        float sacc[4][4];
#pragma unroll
        for (int n = 0; n < 4; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.0f;
        // B (keys) addressing: lane -> key (lane/16)*8 + lane%8, dim offset ((lane/8)%2)*8
        const uint32_t kb_addr = kv_base + (uint32_t)(((lane >> 4) * 8 + (lane & 7)) * kPitch + ((lane >> 3) & 1) * 16);
#pragma unroll 4
        for (int ks = 0; ks < kD / 16; ++ks) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(q_addr + ks * 32, a0, a1, a2, a3);
            uint32_t b0, b1, b2, b3, b4, b5, b6, b7;
            ldsm_x4(kb_addr + ks * 32, b0, b1, b2, b3);                 // keys 0-15
            ldsm_x4(kb_addr + 16 * kPitch + ks * 32, b4, b5, b6, b7);   // keys 16-31
            mma16816(sacc[0], a0, a1, a2, a3, b0, b1);
            mma16816(sacc[1], a0, a1, a2, a3, b2, b3);
            mma16816(sacc[2], a0, a1, a2, a3, b4, b5);
            mma16816(sacc[3], a0, a1, a2, a3, b6, b7);
        }
        // mask invalid slots, scale into the log2 domain, online softmax
        float tmax0 = -CUDART_INF_F, tmax1 = -CUDART_INF_F;
#pragma unroll
        for (int n = 0; n < 4; ++n) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int key = n * 8 + q4 * 2 + c;
                const bool v = bars->valid[s][key] != 0;
                sacc[n][c] = v ? sacc[n][c] * a.scale_log2 : -CUDART_INF_F;
                sacc[n][2 + c] = v ? sacc[n][2 + c] * a.scale_log2 : -CUDART_INF_F;
                tmax0 = fmaxf(tmax0, sacc[n][c]);
                tmax1 = fmaxf(tmax1, sacc[n][2 + c]);
            }
        }
        tmax0 = fmaxf(tmax0, __shfl_xor_sync(0xffffffffu, tmax0, 1));
        tmax0 = fmaxf(tmax0, __shfl_xor_sync(0xffffffffu, tmax0, 2));
        tmax1 = fmaxf(tmax1, __shfl_xor_sync(0xffffffffu, tmax1, 1));
        tmax1 = fmaxf(tmax1, __shfl_xor_sync(0xffffffffu, tmax1, 2));
        const float mn0 = fmaxf(m0, tmax0), mn1 = fmaxf(m1, tmax1);
        const float ref0 = mn0 == -CUDART_INF_F ? 0.0f : mn0;
        const float ref1 = mn1 == -CUDART_INF_F ? 0.0f : mn1;
        const float al0 = exp2f(m0 - ref0), al1 = exp2f(m1 - ref1);
        m0 = mn0;
        m1 = mn1;
        float ps0 = 0.0f, ps1 = 0.0f;
        uint32_t pa[2][4];
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            const float p0 = exp2f(sacc[n][0] - ref0), p1 = exp2f(sacc[n][1] - ref0);
            const float p2 = exp2f(sacc[n][2] - ref1), p3 = exp2f(sacc[n][3] - ref1);
            ps0 += p0 + p1;
            ps1 += p2 + p3;
            // A fragment of P for k-step n/2: regs {r0 lo-k, r1 lo-k, r0 hi-k, r1 hi-k}
            pa[n >> 1][(n & 1) * 2 + 0] = pack_bf16(p0, p1);
            pa[n >> 1][(n & 1) * 2 + 1] = pack_bf16(p2, p3);
        }
        l0 = l0 * al0 + ps0;
        l1 = l1 * al1 + ps1;
#pragma unroll
        for (int n = 0; n < 32; ++n) {
            o[n][0] *= al0;
            o[n][1] *= al0;
            o[n][2] *= al1;
            o[n][3] *= al1;
        }
        // O[16 x 256] += P[16 x 32] . V[32 x 256]
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            // V (trans) addressing: lane -> key kk*16 + (lane%8) + ((lane/8)%2)*8, dims +(lane/16)*8
            const uint32_t v_addr = kv_base +
                                    (uint32_t)((kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * kPitch +
                                               (dh * 256 + (lane >> 4) * 8) * 2);
#pragma unroll
            for (int np = 0; np < 16; ++np) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(v_addr + np * 32, b0, b1, b2, b3);
                mma16816(o[2 * np], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b0, b1);
                mma16816(o[2 * np + 1], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b2, b3);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->empty[s]);
    }
    // full row sums
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

    const int h0 = hg * kHG + hb * 16 + g, h1 = h0 + 8;
    if (a.splits == 1) {
        const float inv0 = l0 > 0.0f ? 1.0f / l0 : 0.0f, inv1 = l1 > 0.0f ? 1.0f / l1 : 0.0f;
        uint32_t *out0 = reinterpret_cast<uint32_t *>(a.out + ((size_t)t * a.H + h0) * kDv + dh * 256);
        uint32_t *out1 = reinterpret_cast<uint32_t *>(a.out + ((size_t)t * a.H + h1) * kDv + dh * 256);
#pragma unroll
        for (int n = 0; n < 32; ++n) {
            out0[n * 4 + q4] = pack_bf16(o[n][0] * inv0, o[n][1] * inv0);
            out1[n * 4 + q4] = pack_bf16(o[n][2] * inv1, o[n][3] * inv1);
        }
        if (a.lse && dh == 0 && q4 == 0) {
            a.lse[(size_t)t * a.H + h0] = l0 > 0.0f ? m0 * 0.69314718055994531f + logf(l0) : -CUDART_INF_F;
            a.lse[(size_t)t * a.H + h1] = l1 > 0.0f ? m1 * 0.69314718055994531f + logf(l1) : -CUDART_INF_F;
        }
    } else {
        const size_t base = (((size_t)t * gridDim.x + hg) * a.splits + split) * kHG;
        float *p0 = a.part_o + (base + hb * 16 + g) * kDv + dh * 256;
        float *p1 = p0 + 8 * kDv;
#pragma unroll
        for (int n = 0; n < 32; ++n) {
            reinterpret_cast<float2 *>(p0)[n * 4 + q4] = make_float2(o[n][0], o[n][1]);
            reinterpret_cast<float2 *>(p1)[n * 4 + q4] = make_float2(o[n][2], o[n][3]);
        }
        if (dh == 0 && q4 == 0) {
            a.part_ml[(base + hb * 16 + g) * 2 + 0] = m0;
            a.part_ml[(base + hb * 16 + g) * 2 + 1] = l0;
            a.part_ml[(base + hb * 16 + g + 8) * 2 + 0] = m1;
            a.part_ml[(base + hb * 16 + g + 8) * 2 + 1] = l1;
        }
    }
}

// Merge split partials: block = (head, head group, query row), 128 threads x 4 dims.
__global__ void __launch_bounds__(128) mla_combine_kernel(MlaArgs a) {
    const int hl = blockIdx.x, hg = blockIdx.y, t = blockIdx.z;
    const int h = hg * kHG + hl;
    if (h >= a.H) return;
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

size_t mla_smem_bytes() { return 128 + kQBytes + (size_t)kStages * kStageBytes + sizeof(MlaBars); }
int mla_key_tile() { return kNT; }

cudaError_t launch_sparse_mla_bf16(const MlaArgs &a, cudaStream_t st) {
    const size_t smem = mla_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(sparse_mla_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    const int groups = (a.H + kHG - 1) / kHG;
    sparse_mla_bf16_kernel<<<dim3(groups, a.splits, a.T), kThreads, smem, st>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess || a.splits == 1) return e;
    mla_combine_kernel<<<dim3(kHG, groups, a.T), 128, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace dsa
