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
    const int mpad = npad > 0 ? npad : 8 * NT;
    const int nrow_ctas = Q.njobs * mpad;
    if (int(blockIdx.x) < nrow_ctas) {
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
