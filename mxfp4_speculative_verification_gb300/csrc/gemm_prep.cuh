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
constexpr int kPrepThreadsBs = 256;  // block-scaled layouts
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
// Block-scaled layouts (kernel of gemm_bs.cuh).  Rows are not rescaled
// (xun = 1); a row holding Inf or NaN gets xun = NaN, which turns every
// output of that row into NaN.  Every stage is written whole: k beyond K
// (up to the next 256) gets zero codes and finite factors.
//
// kind 0 (mxf8f6f4): per 32-k block, x = t1 * 2^e1 + t2 * 2^e2, t1, t2 E4M3,
// e1 = (exponent of the block's largest |x|) - 7, so that the largest |t1|
// lies in [128, 256), and e2 likewise for the residual x - t1 * 2^e1; both
// clamped to the UE8M0 range [-127, 127].  A bf16 value has 8 significant
// bits and each term carries 4, so the pair is exact for every element whose
// residual still lies in the E4M3 range of its block (within 2^16 of the
// block maximum); smaller elements keep about 16 bits.
//
// kind 3 (W4A4, mxf4): X quantised by the pack rule, block by block (the
// exponent e with amax <= 6 2^e at its smallest, 0 for an all-zero block;
// each element the nearest E2M1 value of x 2^-e, ties to the even code):
// one term, the MX-FP4 image of X itself.  A row whose largest |x| is
// below 1 is first scaled up by 2^sh as for kind 1 (never down), which
// keeps the tensor core's block products clear of fp32's subnormal range;
// the rule commutes with that exactly once the rule's clamp of e at -127
// is applied as e >= sh - 127 in the scaled row: the same codes, every
// block exponent shifted by sh.
//
// kind 1 (mxf4): each row is first multiplied by 2^sh, which puts its
// largest |x| in [1, 2) (xun = 2^-sh undoes it), so that the term scales
// below stay inside UE8M0's range for any row; then per 32-k block six E2M1
// terms x = sum t_i * 2^e_i, each the residual of the previous ones rounded
// to nearest (ties to even) at the scale e_i = ceil(log2(max|residual| / 6)),
// which maps the largest residual into (3, 6], E2M1's top binade.  Each term
// leaves at most a quarter of the block's largest residual, so six leave at
// most max|x| / 4^6.
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

// ceil(log2(v / 6)) for v >= 0, clamped to [-127, 127]: v * 2^-e lies in (3, 6]
__device__ __forceinline__ int e2m1_block_exp(float v) {
    const uint32_t b = __float_as_uint(v);
    const int ef = int((b >> 23) & 0xFFu);
    if (ef == 0) return -127;  // zero or subnormal: the smallest scale
    const int e = ef - 127 - 2 + ((b & 0x7FFFFFu) > 0x400000u ? 1 : 0);
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

// 8 values -> 8 E2M1 codes of v * inv, rounded to nearest even (one word,
// element 0 in the low nibble of byte 0)
__device__ __forceinline__ uint32_t e2m1x8(const float (&v)[8], float inv) {
    uint32_t o;
    asm("{\n .reg .b8 b0, b1, b2, b3;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
        " mov.b32 %0, {b0, b1, b2, b3};\n}\n"
        : "=r"(o)
        : "f"(v[0] * inv), "f"(v[1] * inv), "f"(v[2] * inv), "f"(v[3] * inv), "f"(v[4] * inv),
          "f"(v[5] * inv), "f"(v[6] * inv), "f"(v[7] * inv));
    return o;
}

__device__ __forceinline__ void e2m1x8_decode(uint32_t w, float (&v)[8]) {
    uint32_t h[4];
    e2m1x8_to_f16x2x4(w, h[0], h[1], h[2], h[3]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __half2float(__ushort_as_half(uint16_t(h[i] & 0xFFFFu)));
        v[2 * i + 1] = __half2float(__ushort_as_half(uint16_t(h[i] >> 16)));
    }
}

// The smallest E4M3 value >= v for 0 <= v <= 448, and its byte (a UE4M3
// factor: positive E4M3 bytes are ordered like their values).
__device__ __forceinline__ uint32_t ue4m3_ceil(float v, float& value) {
    uint32_t b = e4m3x2_rn(v, 0.f) & 0xFFu;
    float lo, hi;
    e4m3x2_decode(b, lo, hi);
    if (lo < v && b < 0x7Eu) {
        ++b;
        e4m3x2_decode(b, lo, hi);
    }
    value = lo;
    return b;
}

// Byte of B column n's factor for block j of group g in a stage's factor area.
__device__ __forceinline__ int bs_sfb_offset(int n, int g, int j, int copies) {
    return (g * copies + (n >> 7)) * kBsCopyBytes + 16 * (n & 31) + 4 * ((n & 127) >> 5) + j;
}

// Row m of a pass (m >= M: a zero padding row).  Each thread takes 8
// consecutive k; the four threads of a 32-k block are consecutive lanes.
template <int KIND>
__device__ void prep_bs_row(const uint16_t* __restrict__ x, uint8_t* __restrict__ xs,
                            float* __restrict__ xun, int K, int m, int M, int npad) {
    __shared__ int s_bad;
    __shared__ uint32_t s_max;
    if (threadIdx.x == 0) {
        s_bad = 0;
        s_max = 0;
    }
    __syncthreads();
    const uint16_t* row = x + int64_t(m) * K;
    const bool vec = (reinterpret_cast<uintptr_t>(row) & 15) == 0;
    const int nchunks = K / 8;
    float rsc = 1.f, run = 1.f;  // row scale 2^sh and its inverse (mxf4, mxf4nvf4, W4A4)
    int shr = 0;                 // sh itself
    if (KIND >= 1 && m < M) {
        uint32_t mx = 0;  // largest |x| of the row, as bf16 bits (NaN and Inf above every finite)
        for (int k = threadIdx.x; k < K; k += blockDim.x) mx = max(mx, uint32_t(row[k] & 0x7FFFu));
        for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if ((threadIdx.x & 31) == 0) atomicMax(&s_max, mx);
        __syncthreads();
        const int ef = int(s_max >> 7);  // biased exponent of the row's largest |x|
        // the largest |x| into [1, 2) (mxf4), or into [2^10, 2^11) (mxf4nvf4:
        // the first term's UE4M3 factor, max / 6, stays below 448 and the
        // fourth's well above its smallest value)
        if (ef >= 1 && ef <= 254) {
            const int sh = KIND == 3 ? max(127 - ef, 0) : min(KIND == 2 ? 137 - ef : 127 - ef, 127);
            rsc = pow2f_exact(sh);
            run = pow2f_exact(-sh);
            shr = sh;
        } else if (ef == 0 && s_max != 0) {  // a row of subnormals (below 2^-126): into the normal range
            const int sh = KIND == 2 ? 127 : 64;
            rsc = pow2f_exact(sh);
            run = pow2f_exact(-sh);
            shr = sh;
        }
    }
    const int nst = (K + 255) / 256;
    const int bbytes = bs_bstage_bytes(KIND, npad);
    const int brows = bs_brows_bytes(KIND, npad);
    const int copies = bs_sfb_copies(KIND, npad);
    bool bad = false;
    // every chunk of every stage; blockDim.x is a multiple of 32 and of 4 chunks
    for (int base = 0; base < nst * 32; base += int(blockDim.x)) {
        const int c = base + int(threadIdx.x);
        if (base + 32 * (int(threadIdx.x) >> 5) >= nst * 32) break;  // whole warps only (shuffles)
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
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            bad |= !isfinite(f[j]);
            if (KIND >= 1) f[j] *= rsc;  // exact: a power of two, no overflow below the row's maximum
        }
        const int k0 = 8 * c;
        const int st = k0 >> 8;
        const int g = (k0 >> 7) & 1, j = (k0 >> 5) & 3;  // factor group and byte of this block
        uint8_t* stage = xs + int64_t(st) * bbytes;
        uint8_t* sfb = stage + brows;
        const bool lead = (c & 3) == 0;
        if constexpr (KIND == 0) {
            float amax = 0.f;
#pragma unroll
            for (int q = 0; q < 8; ++q) amax = fmaxf(amax, fabsf(f[q]));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            const int e1 = block_exp(amax);
            const uint2 t1 = e4m3x8(f, pow2f_exact(-e1));
            float d[8];
            e4m3x8_decode(t1, d);
            const float s1 = pow2f_exact(e1);
            float rmax = 0.f;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                f[q] = __fsub_rn(f[q], d[q] * s1);  // exact
                rmax = fmaxf(rmax, fabsf(f[q]));
            }
            rmax = fmaxf(rmax, __shfl_xor_sync(0xffffffffu, rmax, 1));
            rmax = fmaxf(rmax, __shfl_xor_sync(0xffffffffu, rmax, 2));
            const int e2 = block_exp(rmax);
            const uint2 t2 = e4m3x8(f, pow2f_exact(-e2));
            const int ch = (k0 >> 7) & 1, u = (k0 >> 4) & 7, half = (k0 >> 3) & 1;
            // B row m holds t1 of X row m, row npad + m its t2 (both rows swizzle alike: npad % 8 == 0)
            uint8_t* sb = stage + ch * (2 * npad * 128);
            const int unit = ((u ^ (m & 7)) << 4) + 8 * half;
            *reinterpret_cast<uint2*>(sb + m * 128 + unit) = act ? t1 : make_uint2(0u, 0u);
            *reinterpret_cast<uint2*>(sb + (npad + m) * 128 + unit) = act ? t2 : make_uint2(0u, 0u);
            if (lead) {
                sfb[bs_sfb_offset(m, g, j, copies)] = act ? uint8_t(e1 + 127) : uint8_t(127);
                sfb[bs_sfb_offset(npad + m, g, j, copies)] = act ? uint8_t(e2 + 127) : uint8_t(127);
            }
        } else if constexpr (KIND == 2) {
            // 8 codes = 4 bytes of the stage's 128-byte row segment; a 16-k block is
            // this lane and its neighbour (c ^ 1), one factor per block and term
            const int b = (k0 & 255) >> 1;
            const int unit = (((b >> 4) ^ (m & 7)) << 4) + (b & 15);
            const int blk = (k0 & 255) >> 4;  // 16-k block of the stage: group blk / 4 (one MMA), byte blk % 4
            const bool lead16 = (c & 1) == 0;
#pragma unroll 1
            for (int t = 0; t < kBsNvTerms; ++t) {
                float amax = 0.f;
#pragma unroll
                for (int q = 0; q < 8; ++q) amax = fmaxf(amax, fabsf(f[q]));
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                float s = 0.f;
                const uint32_t sbyte = ue4m3_ceil(amax * (1.f / 6.f), s);
                const uint32_t codes = act && s > 0.f ? e2m1x8(f, 1.f / s) : 0u;
                float d[8];
                e2m1x8_decode(codes, d);
#pragma unroll
                for (int q = 0; q < 8; ++q) f[q] = __fsub_rn(f[q], d[q] * s);
                const int n = t * npad + m;  // B row (npad % 16 == 0: the same swizzle as row m)
                *reinterpret_cast<uint32_t*>(stage + n * 128 + unit) = codes;
                if (lead16) sfb[bs_sfb_offset(n, blk >> 2, blk & 3, copies)] = act ? uint8_t(sbyte) : uint8_t(0x38);
            }
        } else {
            // 8 codes = 4 bytes of the stage's 128-byte row segment (W4A4:
            // one term, the pack rule itself: e >= -127 before the row
            // scale, an all-zero block gets e = 0)
            const int b = (k0 & 255) >> 1;
            const int unit = (((b >> 4) ^ (m & 7)) << 4) + (b & 15);
            constexpr int kTerms = KIND == 3 ? 1 : kBsF4Terms;
#pragma unroll 1
            for (int t = 0; t < kTerms; ++t) {
                float amax = 0.f;
#pragma unroll
                for (int q = 0; q < 8; ++q) amax = fmaxf(amax, fabsf(f[q]));
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
                const int e = KIND != 3     ? e2m1_block_exp(amax)
                              : amax > 0.f ? max(e2m1_block_exp(amax), shr - 127)
                                           : 0;
                const uint32_t codes = act ? e2m1x8(f, pow2f_exact(-e)) : 0u;
                float d[8];
                e2m1x8_decode(codes, d);
                const float s = pow2f_exact(e);
#pragma unroll
                for (int q = 0; q < 8; ++q) f[q] = __fsub_rn(f[q], d[q] * s);
                const int n = t * npad + m;  // B row (npad % 16 == 0: the same swizzle as row m)
                *reinterpret_cast<uint32_t*>(stage + n * 128 + unit) = codes;
                if (lead) sfb[bs_sfb_offset(n, g, j, copies)] = act ? uint8_t(e + 127) : uint8_t(127);
            }
        }
    }
    if (bad) s_bad = 1;
    __syncthreads();
    if (threadIdx.x == 0) xun[m] = m < M ? (s_bad ? __int_as_float(0x7FC00000) : run) : 0.f;
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
    int bs_npad;          // > 0: X terms + block scales for the block-scaled kernel, this many rows
    int bs_kind;          // its kind: 0 = two E4M3 terms (mxf8f6f4), 1 = six E2M1 terms (mxf4),
                          // 2 = four E2M1 terms with UE4M3 factors per 16 k (mxf4nvf4),
                          // 3 = X quantised by the pack rule, one E2M1 term (W4A4, mxf4)
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
        if (Q.bs_kind == 2)
            prep_bs_row<2>(J.x, reinterpret_cast<uint8_t*>(J.xf), J.xun, J.K, blockIdx.x % mpad, M, Q.bs_npad);
        else if (Q.bs_kind == 3)
            prep_bs_row<3>(J.x, reinterpret_cast<uint8_t*>(J.xf), J.xun, J.K, blockIdx.x % mpad, M, Q.bs_npad);
        else if (Q.bs_kind)
            prep_bs_row<1>(J.x, reinterpret_cast<uint8_t*>(J.xf), J.xun, J.K, blockIdx.x % mpad, M, Q.bs_npad);
        else
            prep_bs_row<0>(J.x, reinterpret_cast<uint8_t*>(J.xf), J.xun, J.K, blockIdx.x % mpad, M, Q.bs_npad);
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
        for (int i = threadIdx.x; i < Q.ncounters; i += int(blockDim.x)) Q.counters[i] = 0;
    } else if (Q.repack_ctas > 0) {
        // realign scale rows: sc_out[n][0..sc_pitch) = sc_in[n][0..nblk), zero padded
        const int64_t total = Q.N * Q.sc_pitch;
        const int64_t stride = int64_t(Q.repack_ctas) * blockDim.x;
        for (int64_t i = int64_t(blockIdx.x - nrow_ctas - 1) * blockDim.x + threadIdx.x;
             i < total; i += stride) {
            const int64_t n = i / Q.sc_pitch;
            const int c = int(i - n * Q.sc_pitch);
            Q.sc_out[i] = c < Q.nblk ? Q.sc_in[n * Q.nblk + c] : uint8_t(0);
        }
    }
}
