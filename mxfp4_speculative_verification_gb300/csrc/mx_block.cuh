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

// The 16 nibble bytes of a block, as four little-endian words, into out16:
// one 16-byte store where out16 is 16-byte aligned, else byte stores.
__device__ __forceinline__ void store_block16(uint8_t* __restrict__ out16, const uint32_t (&w)[4]) {
    if ((reinterpret_cast<uintptr_t>(out16) & 15) == 0) {
        *reinterpret_cast<uint4*>(out16) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) out16[j] = uint8_t(w[j >> 2] >> (8 * (j & 3)));
    }
}

// Elements v[k0 .. k0+7] times inv (an exact power of two) as eight E2M1
// codes, element k0 in the low nibble of byte 0: the hardware conversion
// rounds to the nearest grid value with ties to the even code and keeps the
// sign (also of a value that rounds to zero), which is the pack rule; the
// scaled values never exceed 6, so saturation never acts.
__device__ __forceinline__ uint32_t e2m1x8_rn(const float (&v)[32], int k0, float inv) {
    uint32_t o;
    asm("{\n .reg .b8 b0, b1, b2, b3;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
        " mov.b32 %0, {b0, b1, b2, b3};\n}\n"
        : "=r"(o)
        : "f"(v[k0] * inv), "f"(v[k0 + 1] * inv), "f"(v[k0 + 2] * inv), "f"(v[k0 + 3] * inv),
          "f"(v[k0 + 4] * inv), "f"(v[k0 + 5] * inv), "f"(v[k0 + 6] * inv), "f"(v[k0 + 7] * inv));
    return o;
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
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (!finite) {
        *scale = 255;
        store_block16(out16, w);
        return false;
    }
    const int e = mx_block_exp(amax);
    *scale = uint8_t(e + 127);
    const float inv = exact_pow2(-e);
#pragma unroll
    for (int j = 0; j < 4; ++j) w[j] = e2m1x8_rn(v, 8 * j, inv);
    store_block16(out16, w);
    return true;
}

}  // namespace mxs
