// mxfp8.cuh -- the MXFP8 block rule, shared by the standalone quantiser
// (quant.cu) and the MXFP8 indexer's fused query quantisation
// (indexer_topk.cu), so that both produce the same codes bit for bit.
// OCP Microscaling v1.0 conversion ("Day-0 Inference Adaptation and
// Optimization for Hybrid Attention Architectures", §4 Optimization 2, group
// size 32): X = floor(log2(amax)) - 8 (the E4M3 emax), clamped to the E8M0
// range [-127, 127]; elements E4M3(x / 2^X), round to nearest even,
// saturating at +-448; an all-zero block gets scale byte 127 and zero codes.
#pragma once

#include <cuda_fp8.h>
#include <stdint.h>

namespace dsa {

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

// One block of 32 bf16 values (w: 16 words, low half = lower element) to 32
// E4M3 codes (out: 8 words, byte i = element i) and its E8M0 scale byte.
__device__ __forceinline__ uint8_t mxfp8_block(const uint32_t (&w)[16], uint32_t (&out)[8]) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        amax = fmaxf(amax, fabsf(bf16_bits_to_float(w[i] & 0xFFFFu)));
        amax = fmaxf(amax, fabsf(bf16_bits_to_float(w[i] >> 16)));
    }
    if (amax == 0.0f) {
#pragma unroll
        for (int i = 0; i < 8; ++i) out[i] = 0u;
        return 127;
    }
    int X = floor_log2(amax) - 8;
    X = max(-127, min(127, X));
    const float inv = __uint_as_float((uint32_t)(127 - X) << 23);  // 2^-X, exact (X <= 119 for bf16 inputs)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t a = w[2 * i], b = w[2 * i + 1];
        out[i] = (uint32_t)to_e4m3(bf16_bits_to_float(a & 0xFFFFu) * inv) |
                 ((uint32_t)to_e4m3(bf16_bits_to_float(a >> 16) * inv) << 8) |
                 ((uint32_t)to_e4m3(bf16_bits_to_float(b & 0xFFFFu) * inv) << 16) |
                 ((uint32_t)to_e4m3(bf16_bits_to_float(b >> 16) * inv) << 24);
    }
    return (uint8_t)(X + 127);
}

}  // namespace dsa
