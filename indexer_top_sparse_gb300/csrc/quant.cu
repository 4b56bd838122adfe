// quant.cu -- the quantisers of the layered-quantisation scheme ("Day-0
// Inference Adaptation and Optimization for Hybrid Attention Architectures",
// §4 Optimization 2; "Day0 Inference Adaptation and Performance Optimization
// for a Sparse Hybrid Architecture LLM", §3.1):
//   MXFP8 for the index path: every 32 consecutive values share one E8M0
//   scale 2^X, X = floor(log2(amax)) - 8, elements E4M3 (round to nearest even,
//   saturating at +-448); an all-zero block gets scale byte 127.
//   FP8 for the latent KV cache: the 512 latent dims of a row share one fp32
//   scale s = amax / 448 (1 if amax is 0), elements E4M3(x / s); the 64 rope
//   dims stay bf16.  The tile variant gives every 128 latent dims their own
//   scale by the same rule (the per-token-head-tile granularity, same §4).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "kernels.h"
#include "mxfp8.cuh"
#include "ptx.cuh"

namespace dsa {

namespace {

// One thread per block of 32 values (64 bytes of bf16 in, 32 + 1 bytes out).
__global__ void quant_mxfp8_kernel(const uint16_t *__restrict__ x, int64_t n_blocks, uint8_t *__restrict__ q,
                                   uint8_t *__restrict__ e8m0) {
    const int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (blk >= n_blocks) return;
    const uint4 *src = reinterpret_cast<const uint4 *>(x + blk * 32);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 v = __ldg(src + i);
        w[4 * i] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
    }
    uint32_t out[8];
    e8m0[blk] = mxfp8_block(w, out);
    uint4 *dst = reinterpret_cast<uint4 *>(q + blk * 32);
    dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
    dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
}

// A lane's share of a 576-wide bf16 latent row: latent dims 16l..16l+15 and
// rope dims 2l, 2l+1.
struct LatentLane {
    uint4 v0, v1;
    uint32_t rope;
};
__device__ __forceinline__ LatentLane load_latent(const uint16_t *__restrict__ r, int lane) {
    const uint4 *src = reinterpret_cast<const uint4 *>(r + 16 * lane);
    return {__ldg(src), __ldg(src + 1), __ldg(reinterpret_cast<const uint32_t *>(r + 512) + lane)};
}

// FP8 quantisation of one latent row by a whole warp from the lanes' shares.
// kTiles scales per row: the amax is reduced over the 32 / kTiles lanes of a
// tile.  nope_row, rope_row and scale_row point at the row's outputs.
template <int kTiles>
__device__ __forceinline__ void fp8_row_warp(const LatentLane &x, uint8_t *__restrict__ nope_row,
                                             uint16_t *__restrict__ rope_row, float *__restrict__ scale_row,
                                             int lane) {
    static_assert(kTiles == 1 || kTiles == 4, "one scale per row or per 128 dims");
    constexpr int kLanes = 32 / kTiles;
    const uint4 v0 = x.v0, v1 = x.v1;
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        amax = fmaxf(amax, fabsf(bf16_bits_to_float(w[i] & 0xFFFFu)));
        amax = fmaxf(amax, fabsf(bf16_bits_to_float(w[i] >> 16)));
    }
#pragma unroll
    for (int o = kLanes / 2; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t a = w[2 * i], b = w[2 * i + 1];
        out[i] = (uint32_t)to_e4m3(__fdiv_rn(bf16_bits_to_float(a & 0xFFFFu), s)) |
                 ((uint32_t)to_e4m3(__fdiv_rn(bf16_bits_to_float(a >> 16), s)) << 8) |
                 ((uint32_t)to_e4m3(__fdiv_rn(bf16_bits_to_float(b & 0xFFFFu), s)) << 16) |
                 ((uint32_t)to_e4m3(__fdiv_rn(bf16_bits_to_float(b >> 16), s)) << 24);
    }
    reinterpret_cast<uint4 *>(nope_row)[lane] = make_uint4(out[0], out[1], out[2], out[3]);
    reinterpret_cast<uint32_t *>(rope_row)[lane] = x.rope;
    if (lane % kLanes == 0) scale_row[lane / kLanes] = s;
}

// One warp per 576-wide latent row.
template <int kTiles>
__global__ void quant_fp8_rows_kernel(const uint16_t *__restrict__ kv, int64_t rows, uint8_t *__restrict__ nope,
                                      uint16_t *__restrict__ rope, float *__restrict__ scale) {
    const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    fp8_row_warp<kTiles>(load_latent(kv + row * 576, lane), nope + row * 512, rope + row * 64, scale + row * kTiles,
                         lane);
}

// MXFP8 of one 128-wide index key by a whole warp: lane l holds elements
// 4l..4l+3 (v); the 8 lanes of a 32-element block share its scale (the same
// arithmetic as quant_mxfp8_kernel).
__device__ __forceinline__ void mxfp8_key_warp(const uint2 v, uint8_t *__restrict__ q, uint8_t *__restrict__ e8m0,
                                               int lane) {
    const float f[4] = {bf16_bits_to_float(v.x & 0xFFFFu), bf16_bits_to_float(v.x >> 16),
                        bf16_bits_to_float(v.y & 0xFFFFu), bf16_bits_to_float(v.y >> 16)};
    float amax = fmaxf(fmaxf(fabsf(f[0]), fabsf(f[1])), fmaxf(fabsf(f[2]), fabsf(f[3])));
#pragma unroll
    for (int o = 4; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    uint32_t out = 0u;
    uint8_t byte = 127;
    if (amax != 0.0f) {
        int X = floor_log2(amax) - 8;
        X = max(-127, min(127, X));
        byte = (uint8_t)(X + 127);
        const float inv = __uint_as_float((uint32_t)(127 - X) << 23);  // 2^-X, exact for bf16 inputs
        out = (uint32_t)to_e4m3(f[0] * inv) | ((uint32_t)to_e4m3(f[1] * inv) << 8) |
              ((uint32_t)to_e4m3(f[2] * inv) << 16) | ((uint32_t)to_e4m3(f[3] * inv) << 24);
    }
    reinterpret_cast<uint32_t *>(q)[lane] = out;
    if ((lane & 7) == 0) e8m0[lane >> 3] = byte;
}

// Cache append: warp = new token.  Its position is the sequence's
// (seq_lens[b] - new tokens of b + its rank among them); the page table gives
// the physical row, where the index key and the latent row are written in the
// caches' formats (kIdx: 0 bf16, 1 MXFP8; kKv: 0 bf16, 1 FP8 row scale,
// 4 FP8 tile scales).
template <int kIdx, int kKv>
__global__ void __launch_bounds__(256) cache_append_kernel(AppendArgs a) {
    const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (t >= a.T) return;
    // the new rows first: their loads do not depend on the page walk below
    const bool do_k = a.k_new && a.k_cache, do_kv = a.kv_new && a.kv_cache;
    uint2 kx = make_uint2(0u, 0u);
    if (do_k) kx = __ldg(reinterpret_cast<const uint2 *>(a.k_new + t * 128) + lane);
    LatentLane lx{};
    uint4 bx[3] = {};
    if (do_kv) {
        if constexpr (kKv == 0) {
            const uint4 *s4 = reinterpret_cast<const uint4 *>(a.kv_new + t * 576);
#pragma unroll
            for (int i = 0; i < 3; ++i)
                if (lane + 32 * i < 72) bx[i] = __ldg(s4 + lane + 32 * i);
        } else {
            lx = load_latent(a.kv_new + t * 576, lane);
        }
    }
    int lo = 0, hi = a.B - 1;
    while (lo < hi) {  // the sequence whose new tokens include t
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(a.cu_q + mid) <= t) lo = mid;
        else hi = mid - 1;
    }
    const int b = lo;
    const int64_t c0 = __ldg(a.cu_q + b), n_new = __ldg(a.cu_q + b + 1) - c0;
    const int64_t pos = (int64_t)__ldg(a.seq_lens + b) - n_new + (t - c0);
    if (pos < 0) {
        if (lane == 0) report_error(a.err, kErrBadLen);
        return;
    }
    // a position past the sequence's page-table row is a bad page, unread
    const int page = pos / a.page_size < a.max_pages ? __ldg(a.page_table + (int64_t)b * a.max_pages + pos / a.page_size)
                                                     : -1;
    if (page < 0 || (int64_t)page >= a.num_pages) {
        if (lane == 0) report_error(a.err, kErrBadPage);
        return;
    }
    const int64_t row = (int64_t)page * a.page_size + pos % a.page_size;
    if (do_k) {
        if constexpr (kIdx == 0) {
            reinterpret_cast<uint2 *>(static_cast<uint16_t *>(a.k_cache) + row * 128)[lane] = kx;
        } else {
            mxfp8_key_warp(kx, static_cast<uint8_t *>(a.k_cache) + row * 128, a.k_scale + row * 4, lane);
        }
    }
    if (do_kv) {
        if constexpr (kKv == 0) {
            uint4 *d4 = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(a.kv_cache) + row * 576);
#pragma unroll
            for (int i = 0; i < 3; ++i)
                if (lane + 32 * i < 72) d4[lane + 32 * i] = bx[i];
        } else {
            fp8_row_warp<kKv>(lx, static_cast<uint8_t *>(a.kv_cache) + row * 512, a.kv_rope + row * 64,
                              a.kv_scale + row * kKv, lane);
        }
    }
}

template <int kIdx>
cudaError_t launch_append_kv(const AppendArgs &a, int kv_scales, cudaStream_t st) {
    const unsigned grid = (unsigned)((a.T + 7) / 8);
    if (kv_scales == 0) cache_append_kernel<kIdx, 0><<<grid, 256, 0, st>>>(a);
    else if (kv_scales == 1) cache_append_kernel<kIdx, 1><<<grid, 256, 0, st>>>(a);
    else cache_append_kernel<kIdx, 4><<<grid, 256, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant_mxfp8(const uint16_t *x, int64_t n, uint8_t *q, uint8_t *e8m0, cudaStream_t st) {
    const int64_t blocks = n / 32;
    if (blocks == 0) return cudaSuccess;
    quant_mxfp8_kernel<<<(unsigned)((blocks + 255) / 256), 256, 0, st>>>(x, blocks, q, e8m0);
    return cudaGetLastError();
}

cudaError_t launch_quant_fp8_rows(const uint16_t *kv, int64_t rows, uint8_t *nope, uint16_t *rope, float *scale,
                                  cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    quant_fp8_rows_kernel<1><<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(kv, rows, nope, rope, scale);
    return cudaGetLastError();
}

cudaError_t launch_cache_append(const AppendArgs &a, bool idx_mxfp8, int kv_scales, cudaStream_t st) {
    if (a.T == 0) return cudaSuccess;
    return idx_mxfp8 ? launch_append_kv<1>(a, kv_scales, st) : launch_append_kv<0>(a, kv_scales, st);
}

cudaError_t launch_quant_fp8_tiles(const uint16_t *kv, int64_t rows, uint8_t *nope, uint16_t *rope, float *scale,
                                   cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    quant_fp8_rows_kernel<4><<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(kv, rows, nope, rope, scale);
    return cudaGetLastError();
}

}  // namespace dsa
