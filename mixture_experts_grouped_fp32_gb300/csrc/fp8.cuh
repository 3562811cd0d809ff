// fp8.cuh — E4M3 conversion and the row-quantisation arithmetic shared by the FP8 kernels.
//
// Per-row scaling: absmax over the row, inv = 448 / absmax, code = E4M3(value * inv) rounded to
// nearest even with saturation at 448 (cuda_fp8.h's conversion with __NV_SATFINITE), scale =
// absmax / 448; an all-zero row gets inv = scale = 1 (zero codes).
#pragma once

#include <cuda_fp8.h>
#include <stdint.h>

namespace moe {

__device__ __forceinline__ uint8_t to_e4m3(float v) {
    return static_cast<uint8_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

// The two bf16 values packed in a 32-bit word, widened to fp32 (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float absmax8(uint4 p) {
    const uint32_t w[4] = {p.x, p.y, p.z, p.w};
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
    return m;
}

__device__ __forceinline__ float fp8_inv(float amax) { return amax > 0.0f ? 448.0f / amax : 1.0f; }
__device__ __forceinline__ float fp8_scale(float amax) { return amax > 0.0f ? amax / 448.0f : 1.0f; }

// Blockwise scale of a block with absolute maximum amax: the smallest power of two P with
// fl(amax / 448) <= P, at least 2^-126 (so 1/P is a finite power of two), 1 for an all-zero block.
// frexpf / ldexpf are exact; the division is IEEE (no fast-math), so host and device agree.
__device__ __forceinline__ float pow2_block_scale(float amax) {
    if (!(amax > 0.0f)) return 1.0f;
    const float q = amax / 448.0f;
    int e = 0;
    const float m = frexpf(q, &e);
    const float p = (m == 0.5f) ? q : ldexpf(1.0f, e);
    return fmaxf(p, 1.1754943508222875e-38f);  // 2^-126
}

// Eight bf16 values -> eight E4M3 codes (byte i = code of value i).
__device__ __forceinline__ uint2 codes8(uint4 p, float inv) {
    const uint32_t w[4] = {p.x, p.y, p.z, p.w};
    uint32_t o[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t c0 = to_e4m3(bf16_lo(w[i]) * inv), c1 = to_e4m3(bf16_hi(w[i]) * inv);
        o[i >> 1] |= (c0 | (c1 << 8)) << (16 * (i & 1));
    }
    return make_uint2(o[0], o[1]);
}

}  // namespace moe
