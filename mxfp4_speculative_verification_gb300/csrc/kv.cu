// The MX-FP4 KV cache of the verification block, on sm_103a.
//
// "Next-Gen Speculative Decoding and FP4 Quantization Shake Up LLM Inference
// Economics" keeps keys and values in MX-FP4 (its pipeline diagram's "KV
// Cache Memory Pool (FP4)"; "Benchmarks and Real-World Impact", item 2), and
// "Module 11. Speculative Decoding and Quantization" §4 discards the
// unaccepted suffix and its cache entries after acceptance.
//
// One layer's keys (or values) of B sequences: nibbles [B, L, W/2] and E8M0
// scales [B, L, W/32], one row of W values (every head of one position) per
// position, committed lengths lens[B].
//  * append: the verification pass's T = K + 1 rows of sequence b go to
//    positions lens[b] .. lens[b] + T - 1, each 32-block by the pack rule;
//  * commit: lens[b] += n_emitted[b] (at most L): the last committed token's
//    and the accepted drafts' entries stay, the rejected drafts' entries are
//    the discarded suffix, overwritten by the next pass;
//  * dequant: the decoded rows, zero past each sequence's length.
// Element-wise and bandwidth-bound: the append one thread per 32-element
// block.
#include <cuda_fp16.h>

#include "mx_block.cuh"
#include "mxs_device.cuh"
#include "mxs_internal.h"

namespace mxs {

// Read-back: eight lanes per 32-value block, four values a lane (a quad), so
// a warp writes four whole decoded blocks (512 contiguous bytes) per store;
// grid x over chunks of a row (kKvQuads quads a thread), y over rows.
// (The append keeps one thread per block: its block maximum is a register
// reduction, and the 8-lane form with shuffles measured 2.5x slower.)
constexpr int kKvThreads = 256;
constexpr int kKvQuads = 4;

template <typename T>
__device__ __forceinline__ void load_block32(const T* p, float (&v)[32]);
template <>
__device__ __forceinline__ void load_block32<float>(const float* p, float (&v)[32]) {
    const float4* q = reinterpret_cast<const float4*>(p);  // 128-byte rows, 16-byte aligned
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float4 f = __ldg(q + j);
        v[4 * j] = f.x;
        v[4 * j + 1] = f.y;
        v[4 * j + 2] = f.z;
        v[4 * j + 3] = f.w;
    }
}
template <>
__device__ __forceinline__ void load_block32<uint16_t>(const uint16_t* p, float (&v)[32]) {
    const uint4* q = reinterpret_cast<const uint4*>(p);  // 64-byte rows, 16-byte aligned
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint4 u = __ldg(q + j);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            v[8 * j + 2 * h] = __uint_as_float(w[h] << 16);
            v[8 * j + 2 * h + 1] = __uint_as_float(w[h] & 0xFFFF0000u);
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(256)
    mxfp4_kv_append_kernel(const T* __restrict__ kv, int64_t B, int64_t T_, int64_t W, uint8_t* __restrict__ nib,
                           uint8_t* __restrict__ sc, int64_t L, const int32_t* __restrict__ lens, int32_t* status) {
    const int64_t nblk = W / 32;
    const int64_t total = B * T_ * nblk;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t row = i / nblk, blk = i - row * nblk;  // row = b * T + t
        const int64_t b = row / T_, t = row - b * T_;
        const int64_t pos = int64_t(lens[b]) + t;
        if (pos < 0 || pos >= L) {
            if (blk == 0) report(status, MXS_DEV_KV_FULL);
            continue;
        }
        float v[32];
        load_block32<T>(kv + row * W + blk * 32, v);
        const int64_t cell = b * L + pos;
        if (!pack_block32(v, nib + cell * (W / 2) + blk * 16, sc + cell * (W / 32) + blk))
            report(status, MXS_DEV_NONFINITE);
    }
}

__global__ void __launch_bounds__(256)
    spec_kv_commit_kernel(int32_t* __restrict__ lens, const int32_t* __restrict__ n_emitted, int64_t B, int64_t L) {
    for (int64_t b = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; b < B; b += int64_t(gridDim.x) * blockDim.x) {
        const int64_t l = int64_t(lens[b]) + max(n_emitted[b], 0);
        lens[b] = int32_t(l < L ? l : L);
    }
}

__global__ void __launch_bounds__(kKvThreads)
    mxfp4_kv_dequant_kernel(const uint8_t* __restrict__ nib, const uint8_t* __restrict__ sc, int64_t B, int64_t L,
                            int64_t W, const int32_t* __restrict__ lens, float* __restrict__ out) {
    const int64_t cells = B * L, nq = W / 4;
    for (int64_t cell = blockIdx.y; cell < cells; cell += gridDim.y) {  // cell = b * L + l
        const int64_t b = cell / L, l = cell - b * L;
        const bool live = l < lens[b];
#pragma unroll
        for (int j = 0; j < kKvQuads; ++j) {
            const int64_t q = (int64_t(blockIdx.x) * kKvQuads + j) * kKvThreads + threadIdx.x;
            if (q >= nq) continue;
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
            if (live) {
                const uint16_t two = __ldg(reinterpret_cast<const uint16_t*>(nib + cell * (W / 2) + 2 * q));
                float s, unused;
                e8m0x2_to_f32x2(uint32_t(__ldg(sc + cell * (W / 32) + q / 8)), s, unused);
                uint32_t h0, h1;
                asm("{\n"
                    " .reg .b8 b0, b1;\n"
                    " mov.b16 {b0, b1}, %2;\n"
                    " cvt.rn.f16x2.e2m1x2 %0, b0;\n"
                    " cvt.rn.f16x2.e2m1x2 %1, b1;\n"
                    "}\n"
                    : "=r"(h0), "=r"(h1)
                    : "h"(two));
                const float2 p0 = __half22float2(*reinterpret_cast<const __half2*>(&h0));
                const float2 p1 = __half22float2(*reinterpret_cast<const __half2*>(&h1));
                o = make_float4(p0.x * s, p0.y * s, p1.x * s, p1.y * s);
            }
            *reinterpret_cast<float4*>(out + cell * W + 4 * q) = o;
        }
    }
}

static dim3 kv_grid(int64_t rows, int64_t W) {
    const int64_t per_cta = int64_t(kKvThreads) * kKvQuads;
    const int64_t gx = (W / 4 + per_cta - 1) / per_cta;
    return dim3(unsigned(gx), unsigned(rows < 65535 ? rows : 65535), 1);
}

static unsigned grid_for(int64_t total) {
    const int64_t want = (total + 255) / 256;
    return unsigned(want < 65535 * 16 ? (want > 0 ? want : 1) : 65535 * 16);
}

cudaError_t kv_append_run(const void* kv, int kv_dtype, int64_t B, int64_t T, int64_t W, uint8_t* nibbles,
                          uint8_t* scales, int64_t L, const int32_t* lens, int32_t* dev_status, cudaStream_t stream) {
    const int64_t total = B * T * (W / 32);
    if (total == 0) return cudaSuccess;
    if (kv_dtype == MXS_F32)
        mxfp4_kv_append_kernel<float><<<grid_for(total), 256, 0, stream>>>(static_cast<const float*>(kv), B, T, W,
                                                                           nibbles, scales, L, lens, dev_status);
    else
        mxfp4_kv_append_kernel<uint16_t><<<grid_for(total), 256, 0, stream>>>(
            static_cast<const uint16_t*>(kv), B, T, W, nibbles, scales, L, lens, dev_status);
    return cudaGetLastError();
}

cudaError_t kv_commit_run(int32_t* lens, const int32_t* n_emitted, int64_t B, int64_t L, cudaStream_t stream) {
    if (B == 0) return cudaSuccess;
    spec_kv_commit_kernel<<<grid_for(B), 256, 0, stream>>>(lens, n_emitted, B, L);
    return cudaGetLastError();
}

cudaError_t kv_dequant_run(const uint8_t* nibbles, const uint8_t* scales, int64_t B, int64_t L, int64_t W,
                           const int32_t* lens, float* out, cudaStream_t stream) {
    const int64_t total = B * L * (W / 32);
    if (total == 0) return cudaSuccess;
    mxfp4_kv_dequant_kernel<<<kv_grid(B * L, W), kKvThreads, 0, stream>>>(nibbles, scales, B, L, W, lens, out);
    return cudaGetLastError();
}

}  // namespace mxs
