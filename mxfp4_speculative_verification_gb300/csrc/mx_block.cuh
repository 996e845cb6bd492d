// One 32-element MX-FP4 block by the library's pack rule, shared by
// mxfp4_pack and the KV-cache append ("Module 11. Speculative Decoding and
// Quantization", §12-§13): e = the smallest integer with amax <= 6 * 2^e
// (clamped to [-127, 127]; an all-zero block gets e = 0), each element the
// nearest E2M1 grid value of w / 2^e with ties to the even fraction bit and
// the sign bit kept; a block holding Inf or NaN gets scale byte 255 and zero
// nibbles.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace mxs {

__device__ __forceinline__ float exact_pow2(int e) {  // e in [-149, 127]
    if (e >= -126) return __uint_as_float(uint32_t(e + 127) << 23);
    return __uint_as_float(1u << (e + 149));
}

// Grid code (0..7) of a in [0, 6]: count of decision boundaries passed.
// Midpoints 0.25, 1.25, 2.5, 5 tie to the lower (even) code, midpoints
// 0.75, 1.75, 3.5 tie to the upper (even) code.
__device__ __forceinline__ uint32_t e2m1_magnitude_code(float a) {
    return uint32_t(a > 0.25f) + uint32_t(a >= 0.75f) + uint32_t(a > 1.25f) +
           uint32_t(a >= 1.75f) + uint32_t(a > 2.5f) + uint32_t(a >= 3.5f) + uint32_t(a > 5.0f);
}

// The block exponent of a finite block with largest magnitude amax: the
// smallest integer e with amax <= 6 * 2^e, clamped to [-127, 127]; 0 for an
// all-zero block.
__device__ __forceinline__ int mx_block_exp(float amax) {
    if (!(amax > 0.f)) return 0;
    const uint32_t bits = __float_as_uint(amax);
    const int ex = int(bits >> 23);
    const uint32_t man = bits & 0x7FFFFFu;
    const int e = (ex == 0) ? -127 : ex - 129 + (man > 0x400000u ? 1 : 0);
    return max(-127, min(127, e));
}

// Packs v[0..31] into 16 nibble bytes (element k in byte k/2, even k in the
// low nibble) and one E8M0 byte.  Returns false for a non-finite block.
__device__ __forceinline__ bool pack_block32(const float (&v)[32], uint8_t* __restrict__ out16,
                                             uint8_t* __restrict__ scale) {
    float amax = 0.f;
    bool finite = true;
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        const float a = fabsf(v[k]);
        if (!(a <= 3.402823466e38f)) finite = false;  // Inf or NaN
        else amax = fmaxf(amax, a);
    }
    if (!finite) {
        *scale = 255;
#pragma unroll
        for (int k = 0; k < 16; ++k) out16[k] = 0;
        return false;
    }
    const int e = mx_block_exp(amax);
    *scale = uint8_t(e + 127);
    const float inv = exact_pow2(-e);
#pragma unroll
    for (int k = 0; k < 32; k += 2) {
        const uint32_t c0 = e2m1_magnitude_code(fabsf(v[k]) * inv) | ((__float_as_uint(v[k]) >> 31) << 3);
        const uint32_t c1 = e2m1_magnitude_code(fabsf(v[k + 1]) * inv) | ((__float_as_uint(v[k + 1]) >> 31) << 3);
        out16[k / 2] = uint8_t(c0 | (c1 << 4));
    }
    return true;
}

}  // namespace mxs
