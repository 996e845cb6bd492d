// Device-side definitions shared by the verify-GEMM kernels, included by gemm.cu
// inside namespace mxs: stage geometry, the per-launch problem table, TMA
// helpers and the work-item arithmetic.

constexpr int kStageBlocks = 16;                 // 16 MX blocks = 512 k per stage
constexpr int kBoxBytes = 128;                   // inner extent of one nibble box (256 k)
constexpr int kFragBytesPerBlockTile = 512;      // one 32-k block x 8 rows of X as fp16 fragments

// One GEMM of a launch.  Tensor maps first: they need 64-byte alignment.
struct Problem {
    CUtensorMap tm_w;      // nibbles [N, K/2]: boxes of 128 B x BN rows, 128-byte swizzle
    CUtensorMap tm_s;      // scales [N, nblk] (16-byte row pitch): boxes of 16 B x BN rows
    const uint16_t* xf;    // X fragments [nblk][NT][32 lanes][8 fp16]
    const float* xun;      // [8*NT] per-row unscale
    float* y;              // [M, N]
    float* part;           // split-K partial tiles [ntiles*nsplit][M][BN]
    int* counters;         // split-K arrival counters [ntiles]
    int64_t N;
    int nblk;              // K / 32
    int ntiles;
    int nsplit;
    int stages_per_split;
    int item_begin;        // first work item of this GEMM within the launch
    int sc_from_prep;      // scales were realigned by the preparation kernel
    const uint8_t* sc;     // the scale rows that tm_s streams (row pitch sc_pitch bytes)
    int64_t sc_pitch;
    float gscale;          // NVFP4: the tensor's FP32 scale (unused for MXFP4)
};

// The GEMMs of one launch (a kernel parameter, read in place).  They share
// the row count M of X and are independent of one another.
template <int G>
struct ProblemSet {
    Problem p[G];
    int count;
    int items;  // total work items
    int M;
    int32_t* status;
    int* sched;  // item claim counter, zeroed before the launch (null: static round robin)
    int nstatic; // items each CTA takes in round-robin order before it claims
    int ring;    // block-scaled kernel: stage slots
    // mma.sync kernel, tests of the bounded waits only: the wait limit (ns),
    // and a stage that CTA 0's producer leaves out entirely (-1: none)
    unsigned long long wait_ns;
    int skip_stage;
    // block-scaled kernel, single GEMM without a K split: Y [M, N] as bytes
    // (rows N * 4 apart), written by tensor stores of 16 x 32 boxes when set
    int y_tma;
    CUtensorMap tm_y;
};

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                       uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Sum of the n <= 32 split-K partials p[0], p[stride], ... added in index
// order (the order fixes the result's bits); the loads go out 8 at a time so
// their L2 round trips overlap.
__device__ __forceinline__ float sum_partials(const float* p, int64_t stride, int n) {
    float s = 0.f;
    for (int q0 = 0; q0 < n; q0 += 8) {
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = q0 + j < n ? __ldcg(p + int64_t(q0 + j) * stride) : 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (q0 + j < n) s += v[j];
    }
    return s;
}

struct ItemRange {
    int tile, split, kb0, kb1, nst;
};

__device__ __forceinline__ ItemRange item_range(const Problem& P, int w) {
    ItemRange r;
    r.tile = w % P.ntiles;
    r.split = w / P.ntiles;
    r.kb0 = r.split * P.stages_per_split * kStageBlocks;
    r.kb1 = min(P.nblk, r.kb0 + P.stages_per_split * kStageBlocks);
    r.nst = r.kb1 > r.kb0 ? (r.kb1 - r.kb0 + kStageBlocks - 1) / kStageBlocks : 0;
    return r;
}

// The GEMM that work item w belongs to (binary search over item_begin).
template <int G>
__device__ __forceinline__ int find_problem(const ProblemSet<G>& S, int w) {
    if (G == 1) return 0;
    int lo = 0, hi = S.count - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (S.p[mid].item_begin <= w) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// 2^e as an exact fp32 power of two.
__device__ __forceinline__ float pow2f_exact(int e) {
    // 2^e as fp32 for e in [-149, 127]
    if (e >= -126) return __uint_as_float(uint32_t(e + 127) << 23);
    return __uint_as_float(1u << (e + 149));
}
