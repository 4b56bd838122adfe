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

namespace dsa {

namespace {

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ uint8_t to_e4m3(float v) {
    return (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

// floor(log2(a)) of a positive finite float, subnormals included.
__device__ __forceinline__ int floor_log2(float a) {
    const uint32_t u = __float_as_uint(a);
    const int e = (int)((u >> 23) & 0xFF);
    if (e != 0) return e - 127;
    return (31 - __clz((int)(u & 0x7FFFFF))) - 149;
}

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
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        amax = fmaxf(amax, fabsf(bf16_bits_to_float(w[i] & 0xFFFFu)));
        amax = fmaxf(amax, fabsf(bf16_bits_to_float(w[i] >> 16)));
    }
    uint32_t out[8];
    if (amax == 0.0f) {
        e8m0[blk] = 127;
#pragma unroll
        for (int i = 0; i < 8; ++i) out[i] = 0u;
    } else {
        int X = floor_log2(amax) - 8;
        X = max(-127, min(127, X));
        e8m0[blk] = (uint8_t)(X + 127);
        const float inv = __uint_as_float((uint32_t)(127 - X) << 23);  // 2^-X, exact (X <= 119 for bf16 inputs)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t a = w[2 * i], b = w[2 * i + 1];
            out[i] = (uint32_t)to_e4m3(bf16_bits_to_float(a & 0xFFFFu) * inv) |
                     ((uint32_t)to_e4m3(bf16_bits_to_float(a >> 16) * inv) << 8) |
                     ((uint32_t)to_e4m3(bf16_bits_to_float(b & 0xFFFFu) * inv) << 16) |
                     ((uint32_t)to_e4m3(bf16_bits_to_float(b >> 16) * inv) << 24);
        }
    }
    uint4 *dst = reinterpret_cast<uint4 *>(q + blk * 32);
    dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
    dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
}

// One warp per 576-wide latent row: lane l handles latent dims 16l..16l+15
// and rope dims 2l, 2l+1.  kTiles scales per row: the amax is reduced over
// the 32 / kTiles lanes of a tile.
template <int kTiles>
__global__ void quant_fp8_rows_kernel(const uint16_t *__restrict__ kv, int64_t rows, uint8_t *__restrict__ nope,
                                      uint16_t *__restrict__ rope, float *__restrict__ scale) {
    static_assert(kTiles == 1 || kTiles == 4, "one scale per row or per 128 dims");
    constexpr int kLanes = 32 / kTiles;
    const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const uint16_t *r = kv + row * 576;
    const uint4 *src = reinterpret_cast<const uint4 *>(r + 16 * lane);
    const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
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
    reinterpret_cast<uint4 *>(nope + row * 512)[lane] = make_uint4(out[0], out[1], out[2], out[3]);
    reinterpret_cast<uint32_t *>(rope + row * 64)[lane] = reinterpret_cast<const uint32_t *>(r + 512)[lane];
    if (lane % kLanes == 0) scale[row * kTiles + lane / kLanes] = s;
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

cudaError_t launch_quant_fp8_tiles(const uint16_t *kv, int64_t rows, uint8_t *nope, uint16_t *rope, float *scale,
                                   cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    quant_fp8_rows_kernel<4><<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(kv, rows, nope, rope, scale);
    return cudaGetLastError();
}

}  // namespace dsa
