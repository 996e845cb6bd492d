// The sampling laws acceptance uses, on sm_103a ("Module 11. Speculative
// Decoding and Quantization", §4 "The exact propose-verify-correct cycle":
// temperature, then top-k, then top-p, applied to the target and the draft
// alike; raw probabilities with a filtered law break the proof).
//
// One thread-block cluster of C CTAs x 1024 threads per logit row, the row
// held in registers (16 logits per thread, V <= 131072).  Steps:
//  * the row's largest finite logit m, and whether it holds NaN or +inf (then
//    it has no law);
//  * top-k: the key (monotone uint32 image of the logit) of the k-th largest
//    logit, by a radix select of 4 rounds of 8 bits over token counts;
//    every token with key >= it is kept (ties kept);
//  * top-p: over the kept tokens' masses exp((l - m) / T), the key where the
//    cumulative mass from the top first reaches p, by the same radix select
//    over masses; masses are fixed point (floor(e * 2^46), exact in uint64
//    for any order of addition), so the cut is a deterministic function of
//    the row; ties at the cut are kept;
//  * the kept mass S, and p_t = exp((l_t - m) / T) * 2^46 / S.
// Each round every CTA builds a 256-bin histogram of its slice in shared
// memory; after one cluster barrier every CTA sums the C histograms through
// distributed shared memory and takes the same decision.  Histograms
// alternate between two buffers, so one barrier per round suffices.
#include <cooperative_groups.h>

#include <climits>
#include <cmath>

#include "law.cuh"
#include "mxs_device.cuh"
#include "mxs_internal.h"

namespace cg = cooperative_groups;

namespace mxs {

constexpr int kLawThreads = 1024;
constexpr int kLawChunks = 16;  // logits per thread
constexpr int kLawMaxCluster = 8;
constexpr int64_t kLawSlice = int64_t(kLawThreads) * kLawChunks;
static_assert(kLawMaxV == kLawMaxCluster * kLawSlice, "vocabulary limit");

struct LawArgs {
    const float* logits;  // [R, V]
    int64_t R, V;
    float inv_t;
    int64_t top_k;        // 0 or >= V: no top-k
    float top_p;          // >= 1: no top-p
    LawStats* stats;      // [R] or null
    float* probs;         // [R, V] or null
    int32_t* status;
};

struct LawPub {  // what each CTA publishes to its cluster once
    float m;
    int bad;
    unsigned long long w;
};

__global__ void __launch_bounds__(kLawThreads, 1) sampling_law_kernel(const LawArgs A) {
    __shared__ unsigned long long hist[2][256];
    __shared__ unsigned long long scan_w[8];
    __shared__ float red_m[32];
    __shared__ int red_b[32];
    __shared__ unsigned long long red_w[32];
    __shared__ LawPub pub;
    __shared__ int sel_first, sel_last;
    __shared__ unsigned long long sel_above, sel_bin, sel_total;

    cg::cluster_group cluster = cg::this_cluster();
    const int C = int(cluster.num_blocks());
    const int rank = int(cluster.block_rank());
    const int64_t r = blockIdx.x / C;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t V = A.V;
    const float* row = A.logits + r * V;
    const int64_t v0 = int64_t(rank) * kLawSlice;

    // ---- the slice into registers (element v0 + i * 1024 + tid)
    float x[kLawChunks];
    float mx = -INFINITY;
    int bad = 0;
#pragma unroll
    for (int i = 0; i < kLawChunks; ++i) {
        const int64_t idx = v0 + int64_t(i) * kLawThreads + tid;
        x[i] = idx < V ? __ldg(row + idx) : -INFINITY;
        if (idx < V) {
            if (isnan(x[i]) || x[i] == INFINITY) bad = 1;
            else mx = fmaxf(mx, x[i]);
        }
    }
    auto valid = [&](int i) { return v0 + int64_t(i) * kLawThreads + tid < V; };

    // ---- m and the row's validity across the cluster
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        bad |= __shfl_xor_sync(0xffffffffu, bad, o);
    }
    if (lane == 0) {
        red_m[warp] = mx;
        red_b[warp] = bad;
    }
    __syncthreads();
    if (tid == 0) {
        float a = -INFINITY;
        int b = 0;
        for (int w = 0; w < kLawThreads / 32; ++w) {
            a = fmaxf(a, red_m[w]);
            b |= red_b[w];
        }
        pub.m = a;
        pub.bad = b;
    }
    cluster.sync();
    float m = -INFINITY;
    bad = 0;
    for (int c = 0; c < C; ++c) {
        const LawPub* o = cluster.map_shared_rank(&pub, c);
        m = fmaxf(m, o->m);
        bad |= o->bad;
    }
    LawStats st;
    st.m = m;
    st.cut = 0;
    st.inv_s = 0.f;
    st.ok = !bad && m > -INFINITY;
    const float inv_t = A.inv_t;

    int round = 0;  // alternates the histogram buffers
    // One radix-select pass over the keys >= lo: the largest key K with
    // weight(key >= K) >= target (the weights of valid tokens being 1, or
    // their fixed-point masses).  Returns K; *above gets weight(key > K), and
    // *at weight(key == K).  A target of 0 means "the full weight" (mass
    // pass: the target is taken from the first round's total as ceil(p * W)).
    auto select = [&](bool by_mass, uint32_t lo, unsigned long long target, unsigned long long* above,
                      unsigned long long* at) -> uint32_t {
        uint32_t prefix = 0;
        unsigned long long acc_above = 0;
        for (int rr = 0; rr < 4; ++rr, ++round) {
            const int shift = 24 - 8 * rr;
            unsigned long long* h = hist[round & 1];
            if (tid < 256) h[tid] = 0;
            __syncthreads();
#pragma unroll
            for (int i = 0; i < kLawChunks; ++i) {
                if (!valid(i)) continue;
                const uint32_t k = law_key(x[i]);
                if (k < lo || (rr > 0 && (k >> (shift + 8)) != prefix)) continue;
                const unsigned long long w = by_mass ? law_mass(law_exp(x[i], m, inv_t)) : 1ull;
                if (w) atomicAdd(h + ((k >> shift) & 255u), w);
            }
            __syncthreads();
            cluster.sync();
            // thread t < 256 takes bin 255 - t: an inclusive scan from the top bin down
            unsigned long long tot = 0, incl = 0;
            if (tid < 256) {
                for (int c = 0; c < C; ++c) tot += cluster.map_shared_rank(h, c)[255 - tid];
                incl = tot;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned long long n = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += n;
                }
                if (lane == 31) scan_w[warp] = incl;
            }
            if (tid == 0) {
                sel_first = INT_MAX;
                sel_last = -1;
            }
            __syncthreads();
            if (tid < 256) {
                for (int w = 0; w < warp; ++w) incl += scan_w[w];
                if (tid == 255 && rr == 0 && by_mass && target == 0) sel_total = incl;
            }
            __syncthreads();
            if (by_mass && target == 0 && rr == 0) {
                // the top-p target from the total kept mass
                target = (unsigned long long)ceil(double(A.top_p) * double(sel_total));
                if (target == 0) target = 1;
            }
            // the first bin (from the top) where the cumulative weight reaches the
            // target; if rounding leaves the target out of reach, the last bin
            // holding any weight (everything under the prefix is kept)
            if (tid < 256 && tot > 0) {
                if (incl >= target) atomicMin(&sel_first, tid);
                atomicMax(&sel_last, tid);
            }
            __syncthreads();
            int s = sel_first != INT_MAX ? sel_first : sel_last;
            if (s < 0) s = 0;
            if (tid == s) {
                sel_above = incl - tot;
                sel_bin = tot;
            }
            __syncthreads();
            prefix = (prefix << 8) | uint32_t(255 - s);
            acc_above += sel_above;
            target -= sel_above;
            if (rr == 3) *at = sel_bin;
            __syncthreads();
        }
        *above = acc_above;
        return prefix;
    };

    if (st.ok) {
        uint32_t cut = 0;
        unsigned long long above = 0, at = 0, S = 0;
        const bool topk = A.top_k > 0 && A.top_k < V;
        const bool topp = A.top_p < 1.f;
        if (topk) cut = select(false, 0u, (unsigned long long)A.top_k, &above, &at);
        if (topp) {
            cut = select(true, cut, 0ull, &above, &at);
            S = above + at;
        } else {
            // the kept mass, one cluster reduction
            unsigned long long w = 0;
#pragma unroll
            for (int i = 0; i < kLawChunks; ++i)
                if (valid(i) && law_key(x[i]) >= cut) w += law_mass(law_exp(x[i], m, inv_t));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
            if (lane == 0) red_w[warp] = w;
            __syncthreads();
            if (tid == 0) {
                unsigned long long t = 0;
                for (int q = 0; q < kLawThreads / 32; ++q) t += red_w[q];
                pub.w = t;
            }
            cluster.sync();
            for (int c = 0; c < C; ++c) S += cluster.map_shared_rank(&pub, c)->w;
        }
        st.cut = cut;
        st.inv_s = S > 0 ? float(70368744177664.0 / double(S)) : 0.f;
        if (S == 0) st.ok = 0;
    }
    if (!st.ok && rank == 0 && tid == 0) report(A.status, MXS_DEV_NO_LAW);
    if (A.stats && rank == 0 && tid == 0) A.stats[r] = st;
    if (A.probs) {
        float* out = A.probs + r * V;
#pragma unroll
        for (int i = 0; i < kLawChunks; ++i)
            if (valid(i)) out[v0 + int64_t(i) * kLawThreads + tid] = law_value(x[i], st, inv_t);
    }
    cluster.sync();  // no CTA leaves while another may still read its shared memory
}

// Clusters of C CTAs, C = ceil(V / 16384) (1..8), one per row.
static cudaError_t launch_law(const LawArgs& A, cudaStream_t stream) {
    const int C = int((A.V + kLawSlice - 1) / kLawSlice);
    if (A.R < 1) return cudaSuccess;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(unsigned(A.R * C), 1, 1);
    cfg.blockDim = dim3(kLawThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = unsigned(C);
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, sampling_law_kernel, A);
}

static LawArgs law_args(const float* logits, int64_t R, int64_t V, const LawSampling& s, int32_t* status) {
    LawArgs A{};
    A.logits = logits;
    A.R = R;
    A.V = V;
    A.inv_t = 1.0f / s.temperature;
    A.top_k = s.top_k;
    A.top_p = s.top_p;
    A.status = status;
    return A;
}

cudaError_t sampling_law_run(const float* logits, int64_t R, int64_t V, const LawSampling& s, float* probs,
                             int32_t* dev_status, cudaStream_t stream) {
    LawArgs A = law_args(logits, R, V, s, dev_status);
    A.probs = probs;
    return launch_law(A, stream);
}

cudaError_t law_stats_run(const float* logits, int64_t R, int64_t V, const LawSampling& s, LawStats* stats,
                          int32_t* dev_status, cudaStream_t stream) {
    LawArgs A = law_args(logits, R, V, s, dev_status);
    A.stats = stats;
    return launch_law(A, stream);
}

}  // namespace mxs
