// The X preparation kernel of the verify GEMM, included by gemm.cu inside namespace mxs.
//
// ---------------------------------------------------------------------------
// Preparation: X bf16 [M, K] -> fp16 fragments and per-row unscale factors;
// zeroed split-K counters; optional copy of the scale rows into 16-byte
// aligned rows.
//
// Row m is multiplied by 2^sh with sh = 142 - (biased exponent of max|x|),
// which puts max|x| in [2^15, 2^16): fp16 then holds every element within
// 2^29 of the maximum exactly.  The GEMM multiplies its output by 2^-sh.
// ---------------------------------------------------------------------------
constexpr int kPrepThreads = 512;
constexpr int kPrepChunks = 8;  // 16-byte chunks of one X row kept in registers per thread

__device__ __forceinline__ uint32_t max_abs_bf16x2(uint32_t w, uint32_t m) {
    return max(m, max(w & 0x7FFFu, (w >> 16) & 0x7FFFu));
}

// fp16 image of x * 2^sh for two bf16 values (f1 * f2 = 2^sh, both exact)
__device__ __forceinline__ uint32_t scale_bf16x2_to_f16x2(uint32_t w, float f1, float f2) {
    const float lo = (__uint_as_float(w << 16) * f1) * f2;
    const float hi = (__uint_as_float(w & 0xFFFF0000u) * f1) * f2;
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// ---------------------------------------------------------------------------
// Block-scaled layout (kernel of gemm_bs.cuh): per 32-k block of a row,
//   x = t1 * 2^e1 + t2 * 2^e2,  t1, t2 E4M3,
// e1 = (exponent of the block's largest |x|) - 7, so that the largest |t1|
// lies in [128, 256), and e2 likewise for the residual x - t1 * 2^e1; both
// clamped to the UE8M0 range [-127, 127].  A bf16 value has 8 significant
// bits and each term carries 4, so the pair is exact for every element whose
// residual still lies in the E4M3 range of its block (within 2^16 of the
// block maximum); smaller elements keep about 16 bits.  Rows are not
// rescaled (xun = 1); a row holding Inf or NaN gets xun = NaN, which turns
// every output of that row into NaN.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t e4m3x2_rn(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ void e4m3x2_decode(uint32_t two, float& lo, float& hi) {
    uint32_t h2;
    asm("{\n .reg .b16 t;\n cvt.u16.u32 t, %1;\n cvt.rn.f16x2.e4m3x2 %0, t;\n}\n" : "=r"(h2) : "r"(two));
    lo = __half2float(__ushort_as_half(uint16_t(h2 & 0xFFFFu)));
    hi = __half2float(__ushort_as_half(uint16_t(h2 >> 16)));
}

// floor(log2 v) - 7 for v >= 0 (the block exponent), clamped to [-127, 127]
__device__ __forceinline__ int block_exp(float v) {
    const int e = int((__float_as_uint(v) >> 23) & 0xFFu) - 127 - 7;
    return max(-127, min(127, e));
}

// 8 values -> 8 E4M3 codes of v * 2^-e (two little-endian words)
__device__ __forceinline__ uint2 e4m3x8(const float (&v)[8], float inv) {
    uint2 o;
    o.x = e4m3x2_rn(v[0] * inv, v[1] * inv) | (e4m3x2_rn(v[2] * inv, v[3] * inv) << 16);
    o.y = e4m3x2_rn(v[4] * inv, v[5] * inv) | (e4m3x2_rn(v[6] * inv, v[7] * inv) << 16);
    return o;
}

__device__ __forceinline__ void e4m3x8_decode(uint2 c, float (&v)[8]) {
    e4m3x2_decode(c.x & 0xFFFFu, v[0], v[1]);
    e4m3x2_decode(c.x >> 16, v[2], v[3]);
    e4m3x2_decode(c.y & 0xFFFFu, v[4], v[5]);
    e4m3x2_decode(c.y >> 16, v[6], v[7]);
}

// Row m of a pass (m >= M: a zero padding row).  Each thread takes 8
// consecutive k; the four threads of a 32-k block are consecutive lanes.
__device__ void prep_bs_row(const uint16_t* __restrict__ x, uint8_t* __restrict__ xs,
                            float* __restrict__ xun, int K, int m, int M, int npad) {
    __shared__ int s_bad;
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    const uint16_t* row = x + int64_t(m) * K;
    const bool vec = (reinterpret_cast<uintptr_t>(row) & 15) == 0;
    const int nchunks = K / 8;
    const int bbytes = 512 * npad;                        // B rows of one 256-k stage
    uint8_t* sfb = xs + int64_t((K + 255) / 256) * bbytes;  // scale bytes, after all stages
    bool bad = false;
    for (int base = 0; base < nchunks; base += kPrepThreads) {
        const int c = base + int(threadIdx.x);
        const bool act = c < nchunks && m < M;
        float f[8];
        if (act && vec) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(row) + c);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                f[2 * j] = __uint_as_float(w[j] << 16);
                f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] = act ? __uint_as_float(uint32_t(row[8 * c + j]) << 16) : 0.f;
        }
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            bad |= !isfinite(f[j]);
            amax = fmaxf(amax, fabsf(f[j]));
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        const int e1 = block_exp(amax);
        const uint2 t1 = e4m3x8(f, pow2f_exact(-e1));
        float d[8];
        e4m3x8_decode(t1, d);
        const float s1 = pow2f_exact(e1);
        float rmax = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            f[j] = __fsub_rn(f[j], d[j] * s1);  // exact
            rmax = fmaxf(rmax, fabsf(f[j]));
        }
        rmax = fmaxf(rmax, __shfl_xor_sync(0xffffffffu, rmax, 1));
        rmax = fmaxf(rmax, __shfl_xor_sync(0xffffffffu, rmax, 2));
        const int e2 = block_exp(rmax);
        const uint2 t2 = e4m3x8(f, pow2f_exact(-e2));
        if (c < nchunks) {
            const int k0 = 8 * c;
            const int st = k0 >> 8, ch = (k0 >> 7) & 1, u = (k0 >> 4) & 7, half = (k0 >> 3) & 1;
            // B row m holds t1 of X row m, row npad + m its t2 (both rows swizzle alike: npad % 8 == 0)
            uint8_t* sb = xs + int64_t(st) * bbytes + ch * (2 * npad * 128);
            const int unit = ((u ^ (m & 7)) << 4) + 8 * half;
            *reinterpret_cast<uint2*>(sb + m * 128 + unit) = act ? t1 : make_uint2(0u, 0u);
            *reinterpret_cast<uint2*>(sb + (npad + m) * 128 + unit) = act ? t2 : make_uint2(0u, 0u);
            if ((c & 3) == 0) {
                const int j = (k0 >> 5) & 7;
                uint8_t* ss = sfb + int64_t(st) * (16 * npad);
                ss[m * 8 + j] = act ? uint8_t(e1 + 127) : uint8_t(0);
                ss[(npad + m) * 8 + j] = act ? uint8_t(e2 + 127) : uint8_t(0);
            }
        }
    }
    if (bad) s_bad = 1;
    __syncthreads();
    if (threadIdx.x == 0) xun[m] = m < M ? (s_bad ? __int_as_float(0x7FC00000) : 1.f) : 0.f;
}

// One distinct X of a launch.
struct PrepJob {
    const uint16_t* x;  // [M, K] bf16
    uint16_t* xf;       // fragments out
    float* xun;         // [8*NT] unscale factors out
    int K;
};

constexpr int kPrepMaxJobs = 16;

struct PrepSet {
    PrepJob job[kPrepMaxJobs];
    int njobs;
    int M;
    int NT;
    int umma_npad;        // 0: mma.sync fragments; else swizzled tcgen05 tiles of this many rows
    int bs_npad;          // > 0: two E4M3 terms + block scales for the block-scaled kernel, this many rows
    int* counters;        // split-K counters to zero (may be null)
    int ncounters;
    const uint8_t* sc_in;  // scale realignment (single GEMM only; null otherwise)
    int64_t N;
    int nblk;
    int sc_pitch;
    uint8_t* sc_out;
    int repack_ctas;
};

__global__ void __launch_bounds__(kPrepThreads) mxfp4_gemm_prep_kernel(const __grid_constant__ PrepSet Q) {
    pdl_trigger();
    pdl_wait();  // the workspace may still be in use by the previous GEMM
    const int NT = Q.NT, M = Q.M;
    const int npad = Q.umma_npad;
    const int mpad = Q.bs_npad > 0 ? Q.bs_npad : (npad > 0 ? npad : 8 * NT);
    const int nrow_ctas = Q.njobs * mpad;
    if (int(blockIdx.x) < nrow_ctas && Q.bs_npad > 0) {
        const PrepJob& J = Q.job[blockIdx.x / mpad];
        prep_bs_row(J.x, reinterpret_cast<uint8_t*>(J.xf), J.xun, J.K, blockIdx.x % mpad, M, Q.bs_npad);
    } else if (int(blockIdx.x) < nrow_ctas) {
        const PrepJob& J = Q.job[blockIdx.x / mpad];
        const int K = J.K;
        const uint16_t* __restrict__ x = J.x;
        uint16_t* __restrict__ xf = J.xf;
        float* __restrict__ xun = J.xun;
        const int m = blockIdx.x % mpad;
        const int nt = m >> 3, gg = m & 7;
        __shared__ uint32_t smax;
        if (threadIdx.x == 0) smax = 0;
        __syncthreads();
        const uint16_t* row = x + int64_t(m) * K;
        const int nchunks = K / 8;  // 8 consecutive k: one 16-byte piece of a fragment
        const bool fast = (K <= kPrepThreads * kPrepChunks * 8) &&
                          (reinterpret_cast<uintptr_t>(row) % 16 == 0);
        uint4 v[kPrepChunks];
        uint32_t mx = 0;
        if (m < M) {
            if (fast) {
#pragma unroll
                for (int i = 0; i < kPrepChunks; ++i) {
                    const int c = threadIdx.x + i * kPrepThreads;
                    v[i] = c < nchunks ? __ldg(reinterpret_cast<const uint4*>(row) + c)
                                       : make_uint4(0, 0, 0, 0);
                    mx = max_abs_bf16x2(v[i].x, mx);
                    mx = max_abs_bf16x2(v[i].y, mx);
                    mx = max_abs_bf16x2(v[i].z, mx);
                    mx = max_abs_bf16x2(v[i].w, mx);
                }
            } else {
                for (int k = threadIdx.x; k < K; k += kPrepThreads) mx = max(mx, uint32_t(row[k] & 0x7FFFu));
            }
        }
        for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if ((threadIdx.x & 31) == 0) atomicMax(&smax, mx);
        __syncthreads();
        int emax = int(smax >> 7);  // biased exponent of max|x| (NaN/Inf -> 255)
        if (emax < 1) emax = 1;
        const int sh = 142 - emax;  // in [-113, 141]
        const float f1 = pow2f_exact(sh / 2), f2 = pow2f_exact(sh - sh / 2);
        if (threadIdx.x == 0) xun[m] = (m < M) ? pow2f_exact(-sh) : 0.f;
        auto frag = [&](int c) -> uint4* {
            const int k0 = c * 8;
            if (npad > 0) {
                // [stage of 512 k][chunk of 64 k][row][128 B, 16-byte units swizzled by row % 8]
                const int st = k0 >> 9, ch = (k0 >> 6) & 7, u = (k0 >> 3) & 7;
                const int64_t byte = int64_t(st) * npad * 1024 + int64_t(ch) * npad * 128 + m * 128 +
                                     ((u ^ (m & 7)) << 4);
                return reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(xf) + byte);
            }
            const int blk = k0 >> 5, tt = (k0 & 31) >> 3;
            return reinterpret_cast<uint4*>(xf + ((int64_t(blk) * NT + nt) * 32 + gg * 4 + tt) * 8);
        };
        if (m >= M) {  // padding rows of the fragment tile
            for (int c = threadIdx.x; c < nchunks; c += kPrepThreads) *frag(c) = make_uint4(0, 0, 0, 0);
        } else if (fast) {
#pragma unroll
            for (int i = 0; i < kPrepChunks; ++i) {
                const int c = threadIdx.x + i * kPrepThreads;
                if (c >= nchunks) break;
                uint4 o;
                o.x = scale_bf16x2_to_f16x2(v[i].x, f1, f2);
                o.y = scale_bf16x2_to_f16x2(v[i].y, f1, f2);
                o.z = scale_bf16x2_to_f16x2(v[i].z, f1, f2);
                o.w = scale_bf16x2_to_f16x2(v[i].w, f1, f2);
                *frag(c) = o;
            }
        } else {
            for (int c = threadIdx.x; c < nchunks; c += kPrepThreads) {
                uint32_t w[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    w[q] = uint32_t(row[c * 8 + 2 * q]) | (uint32_t(row[c * 8 + 2 * q + 1]) << 16);
                uint4 o;
                o.x = scale_bf16x2_to_f16x2(w[0], f1, f2);
                o.y = scale_bf16x2_to_f16x2(w[1], f1, f2);
                o.z = scale_bf16x2_to_f16x2(w[2], f1, f2);
                o.w = scale_bf16x2_to_f16x2(w[3], f1, f2);
                *frag(c) = o;
            }
        }
    } else if (int(blockIdx.x) == nrow_ctas) {
        for (int i = threadIdx.x; i < Q.ncounters; i += kPrepThreads) Q.counters[i] = 0;
    } else if (Q.repack_ctas > 0) {
        // realign scale rows: sc_out[n][0..sc_pitch) = sc_in[n][0..nblk), zero padded
        const int64_t total = Q.N * Q.sc_pitch;
        const int64_t stride = int64_t(Q.repack_ctas) * kPrepThreads;
        for (int64_t i = int64_t(blockIdx.x - nrow_ctas - 1) * kPrepThreads + threadIdx.x;
             i < total; i += stride) {
            const int64_t n = i / Q.sc_pitch;
            const int c = int(i - n * Q.sc_pitch);
            Q.sc_out[i] = c < Q.nblk ? Q.sc_in[n * Q.nblk + c] : uint8_t(0);
        }
    }
}
