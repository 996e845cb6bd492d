// The sampling laws acceptance uses, on sm_103a ("Module 11. Speculative
// Decoding and Quantization", §4 "The exact propose-verify-correct cycle":
// temperature, then top-k, then top-p, applied to the target and the draft
// alike; raw probabilities with a filtered law break the proof).
//
// Two forms compute the same statistics bit for bit.  Below 128 rows: one
// thread-block cluster of C CTAs x 512 threads per logit row, each CTA
// holding a 16384-logit slice in shared memory (V <= 131072); two CTAs share
// an SM, so one row's barriers overlap another row's work.  From 128 rows:
// one 1024-thread CTA per row that streams the row again for each pass (the
// row form, further down), with about one row per SM in flight.  Steps:
//  * the row's largest finite logit m, and whether it holds NaN or +inf (then
//    it has no law);
//  * top-k: the key (monotone uint32 image of the logit) of the k-th largest
//    logit; every token with key >= it is kept (ties kept);
//  * top-p: over the kept tokens' masses exp((l - m) / T) in fixed point
//    (floor(e * 2^46), exact in uint64 for any order of addition, so the cut
//    is a deterministic function of the row), the key where the cumulative
//    mass from the top first reaches ceil(p * total); ties at the cut kept;
//  * the kept mass S, and p_t = exp((l_t - m) / T) * 2^46 / S.
//
// Each cut (by token count for top-k, by mass for top-p) is found in three
// narrowing steps over tokens ordered by their log-mass a = (l - m) / T,
// which is monotone in the key:
//  1. one pass over the slice sums the weight of four classes, a in (-4, 0],
//     (-8, -4], (-16, -8] and below, in registers; one cluster exchange gives
//     the class where the cumulative weight reaches the target;
//  2. the tokens of that class fill a 512-bin histogram of finer log-mass
//     steps (1/128 nat in the top classes); one exchange gives the bin;
//  3. the tokens of that bin (typically tens) are gathered from every CTA,
//     and each CTA ranks them by key exactly.
// If the bin holds too many tokens to gather, a radix select over its keys
// (4 rounds of 8 bits, one exchange each) finishes instead.  Every step is a
// function of the row alone, so all CTAs of a cluster take the same
// decisions, and the result is the same as one radix select over the row.
// Tokens of zero fixed-point mass (e < 2^-46) may enter the fine histogram
// and the gather of a top-p cut (tokens below the top-k cut never do): they
// add nothing to any sum, and the cut, the largest key whose tokens at or
// above it reach the target, never falls on them.
#include <cooperative_groups.h>

#include <climits>
#include <cmath>
#include <cstdlib>
#include <cstring>

#include "law.cuh"
#include "mxs_device.cuh"
#include "mxs_internal.h"

namespace cg = cooperative_groups;

namespace mxs {

constexpr int kLawThreads = 512;
constexpr int kLawWarps = kLawThreads / 32;
constexpr int kLawChunksWide = 32;  // logits per thread: 16384-logit slices, clusters of up to 8
constexpr int kLawChunksNarrow = 16;  // 8192-logit slices, clusters of up to 16 (few rows)
constexpr int kLawMaxClusterAll = 16;
template <int CH>
constexpr int law_max_cluster() { return int(kLawMaxV / (int64_t(kLawThreads) * CH)); }
constexpr int kLawBins = 512;  // one fine-histogram bin per thread
constexpr int kGatherCap = 128;    // tokens one CTA may contribute to a gather
constexpr int kGatherTotal = 256;  // tokens a cluster may gather
constexpr int kLawVals = 4;        // values one step publishes to the cluster
static_assert(law_max_cluster<kLawChunksWide>() == 8 && law_max_cluster<kLawChunksNarrow>() == kLawMaxClusterAll,
              "vocabulary limit");

struct LawArgs {
    const float* logits;   // rows 0 .. R1-1: [R1, V]
    const float* logits2;  // rows R1 .. R-1: [R - R1, V] (a second tensor, one launch for both)
    int64_t R1;
    int64_t R, V;
    float inv_t;
    int64_t top_k;        // 0 or >= V: no top-k
    float top_p;          // >= 1: no top-p
    LawStats* stats;      // [R] or null
    float* probs;         // [R, V] or null
    int32_t* status;
};

struct GatherEntry {
    uint32_t key;
    float x;
};

// Shared memory of one CTA (dynamic, about 70 KB with 16384-logit slices).
template <int CH>
struct LawSmem {
    float xs[CH * kLawThreads];          // element v0 + i * 512 + t at [i * 512 + t]
    GatherEntry glist[kGatherCap];       // this CTA's tokens of the gathered bin
    GatherEntry gall[kGatherTotal];      // the cluster's, in CTA order
    unsigned long long gw[kGatherTotal]; // and their weights
    unsigned long long red[kLawWarps][kLawVals];
    unsigned long long tot[kLawVals];    // cluster sums
    unsigned long long scan_w[kLawWarps];
    unsigned long long sel_above, sel_at, sel_total;
    int gcount;                          // tokens found for the gather (may exceed the cap)
    int goff[kLawMaxClusterAll + 1];
    int sel_first, sel_last;
    uint32_t sel_key, sel_min;
    int sel_any, sel_idx;
    float pub_m;
    int pub_bad;
    float m;
    int bad;
};

// Log-mass classes of the tokens, by a = (l - m) / T <= 0: 0 for a > -4, 1
// for (-8, -4], 2 for (-16, -8], 3 below.  (On logits like N(0, 3) at T =
// 0.8 the top-p 0.9 cut lies 7 to 9 nats below the maximum.)

// Fine bin of a token within its class (0 holds the largest logits): steps
// of 1/128 nat in classes 0 and 1, 1/64 in class 2, 1/16 in class 3 (bin 511
// also takes every token 48 or more below the maximum).  Monotone in a.
__device__ __forceinline__ int law_fine(float a, int c) {
    const float lo = c == 0 ? 0.f : c == 1 ? 4.f : c == 2 ? 8.f : 16.f;
    const float sc = c <= 1 ? 128.f : c == 2 ? 64.f : 16.f;
    const float f = (-a - lo) * sc;
    return f >= float(kLawBins - 1) ? kLawBins - 1 : int(f);
}

// Sum of a 64-bit value over a warp (two 32-bit shuffles per step).
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

struct LawCut {
    uint32_t key;              // the cut: tokens with key >= it are kept
    unsigned long long above;  // weight of the tokens with larger keys
    unsigned long long at;     // weight of the tokens with this key
};

template <bool B>
struct LawTag {
    static constexpr bool value = B;
};

// One token of the class pass: its weight (1, or its fixed-point mass as two
// 23-bit digits; 0 below the key lo, or for a slot without a token) added to
// the cumulative class sums -- sum 0 over every token, sums 1..3 over the
// tokens with a > -4, -8, -16 -- each digit kept in 32 bits (a digit is at
// most 2^23 and a thread adds at most 128 tokens: at most 2^30).  Returns the
// three comparisons.
template <bool BY_MASS, bool HAS_LO>
__device__ __forceinline__ void class_add(float x, float m, float inv_t, uint32_t lo, bool valid,
                                          uint32_t (&h)[kLawVals], uint32_t (&l)[kLawVals], bool& p4, bool& p8,
                                          bool& p16) {
    const float a = (x - m) * inv_t;
    p4 = a > -4.f;
    p8 = a > -8.f;
    p16 = a > -16.f;
    const bool in = valid && (!HAS_LO || law_key(x) >= lo);
    if constexpr (BY_MASS) {
        uint32_t hb, lb;
        law_mass_digits(in ? law_exp(x, m, inv_t) : 0.f, hb, lb);
        hb -= kMassBias;
        lb -= kMassBias;
        h[0] += hb;
        l[0] += lb;
        if (p4) {
            h[1] += hb;
            l[1] += lb;
        }
        if (p8) {
            h[2] += hb;
            l[2] += lb;
        }
        if (p16) {
            h[3] += hb;
            l[3] += lb;
        }
    } else {
        const uint32_t w = in ? 1u : 0u;
        l[0] += w;
        l[1] += p4 ? w : 0u;
        l[2] += p8 ? w : 0u;
        l[3] += p16 ? w : 0u;
    }
}

// The class sums of one thread as 64-bit weights.
template <bool BY_MASS>
__device__ __forceinline__ void class_sums(const uint32_t (&h)[kLawVals], const uint32_t (&l)[kLawVals],
                                           unsigned long long (&v)[kLawVals]) {
#pragma unroll
    for (int j = 0; j < kLawVals; ++j)
        v[j] = BY_MASS ? (static_cast<unsigned long long>(h[j]) << 23) + l[j] : static_cast<unsigned long long>(l[j]);
}

// The tokens of fine bin f of class c are those whose t = -a lies in [*tlo,
// *thi]: law_fine is non-decreasing in t, so both ends are found by bisection
// over the bit patterns of non-negative floats, with law_fine itself (the
// same float operations as the per-token test they replace).
__device__ inline void fine_bin_range(int c, int f, float* tlo, float* thi) {
    auto first_at_least = [&](int g) {  // smallest t >= 0 with law_fine(-t, c) >= g
        uint32_t lo = 0u, hi = 0x7F800000u;  // +inf lands in bin 511
        while (lo < hi) {
            const uint32_t mid = lo + ((hi - lo) >> 1);
            if (law_fine(-__uint_as_float(mid), c) >= g) hi = mid;
            else lo = mid + 1u;
        }
        return lo;
    };
    *tlo = __uint_as_float(first_at_least(f));
    *thi = f >= kLawBins - 1 ? INFINITY : __uint_as_float(first_at_least(f + 1) - 1u);
}

// Whether a token of log-mass a lies in class c.
__device__ __forceinline__ bool in_class(float a, int c) {
    const float hi = c == 0 ? INFINITY : c == 1 ? -4.f : c == 2 ? -8.f : -16.f;
    const float lo = c == 0 ? -4.f : c == 1 ? -8.f : -16.f;
    return a <= hi && (c == 3 || a > lo);
}

template <int CH>
__global__ void __launch_bounds__(kLawThreads, 2) sampling_law_kernel(const LawArgs A) {
    constexpr int kLawChunks = CH;
    constexpr int64_t kLawSlice = int64_t(kLawThreads) * CH;
    constexpr int kLawMaxCluster = law_max_cluster<CH>();
    extern __shared__ __align__(16) uint8_t law_smem_raw[];
    LawSmem<CH>& S = *reinterpret_cast<LawSmem<CH>*>(law_smem_raw);
    __shared__ uint32_t hist_cnt[2][kLawBins], hist_lo[2][kLawBins], hist_hi[2][kLawBins];
    __shared__ unsigned long long pubv[2][kLawVals];

    cg::cluster_group cluster = cg::this_cluster();
    const int C = int(cluster.num_blocks());
    const int rank = int(cluster.block_rank());
    const int64_t r = blockIdx.x / C;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t V = A.V;
    const int64_t v0 = int64_t(rank) * kLawSlice;
    const int nv = int(V - v0 < kLawSlice ? V - v0 : kLawSlice);  // tokens in this slice, >= 1

    // ---- the slice into shared memory; its largest finite logit, and NaN / +inf
    {
        const float* row = (r < A.R1 ? A.logits + r * V : A.logits2 + (r - A.R1) * V) + v0;
        float mx = -INFINITY;
        int bad = 0;
#pragma unroll
        for (int i = 0; i < kLawChunks; ++i) {
            const int j = i * kLawThreads + tid;
            float v = -INFINITY;
            if (j < nv) {
                v = __ldg(row + j);
                bad |= int(v != v);
                mx = fmaxf(mx, v);  // NaN ignored; +inf makes the row bad below
            }
            S.xs[j] = v;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            bad |= __shfl_xor_sync(0xffffffffu, bad, o);
        }
        if (lane == 0) {
            S.red[warp][0] = __float_as_uint(mx);
            S.red[warp][1] = unsigned(bad);
        }
        __syncthreads();
        if (tid == 0) {
            float a = -INFINITY;
            int b = 0;
            for (int w = 0; w < kLawWarps; ++w) {
                a = fmaxf(a, __uint_as_float(uint32_t(S.red[w][0])));
                b |= int(S.red[w][1]);
            }
            S.pub_m = a;
            S.pub_bad = b;
        }
        cluster.sync();
        if (warp == 0) {
            float a = -INFINITY;
            int b = 0;
            if (lane < C) {
                const LawSmem<CH>* o = cluster.map_shared_rank(&S, lane);
                a = o->pub_m;
                b = o->pub_bad;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
                b |= __shfl_xor_sync(0xffffffffu, b, o);
            }
            if (lane == 0) {
                S.m = a;
                S.bad = b;
            }
        }
        __syncthreads();
    }
    const float m = S.m;
    const float inv_t = A.inv_t;
    LawStats st;
    st.m = m;
    st.cut = 0;
    st.inv_s = 0.f;
    st.ok = !S.bad && m > -INFINITY && m < INFINITY;

    int pb = 0;  // alternates the published-sum buffers
    int hb = 0;  // alternates the histogram buffers
    // Sums of kLawVals values over the cluster, into S.tot (all threads).
    auto cluster_sum = [&](unsigned long long (&v)[kLawVals]) {
#pragma unroll
        for (int j = 0; j < kLawVals; ++j) v[j] = warp_sum_u64(v[j]);
        if (lane == 0)
#pragma unroll
            for (int j = 0; j < kLawVals; ++j) S.red[warp][j] = v[j];
        __syncthreads();
        unsigned long long* pub = pubv[pb];
        pb ^= 1;
        if (tid < kLawVals) {
            unsigned long long t = 0;
            for (int w = 0; w < kLawWarps; ++w) t += S.red[w][tid];
            pub[tid] = t;
        }
        cluster.sync();
        if (tid < kLawVals) {
            unsigned long long t = 0;
            for (int c = 0; c < C; ++c) t += cluster.map_shared_rank(pub, c)[tid];
            S.tot[tid] = t;
        }
        __syncthreads();
    };
    // A fresh CTA histogram; returns its buffer index.
    auto hist_begin = [&]() -> int {
        const int b = hb;
        hb ^= 1;
        if (tid < kLawBins) {
            hist_cnt[b][tid] = 0;
            hist_lo[b][tid] = 0;
            hist_hi[b][tid] = 0;
        }
        __syncthreads();
        return b;
    };
    auto hist_put = [&](int b, int bin, bool by_mass, unsigned long long w) {
        if (!by_mass) {
            atomicAdd(&hist_cnt[b][bin], 1u);
            return;
        }
        const uint32_t lo = uint32_t(w);
        uint32_t hi = uint32_t(w >> 32);
        const uint32_t old = atomicAdd(&hist_lo[b][bin], lo);
        if (old + lo < old) ++hi;
        if (hi) atomicAdd(&hist_hi[b][bin], hi);
    };
    // After every CTA filled buffer b: the cluster's weight at bin tid.
    auto hist_end = [&](int b, bool by_mass) -> unsigned long long {
        __syncthreads();
        cluster.sync();
        unsigned long long t = 0;
        if (tid < kLawBins)
            for (int c = 0; c < C; ++c) {
                if (by_mass) {
                    const uint32_t lo = *cluster.map_shared_rank(&hist_lo[b][tid], c);
                    const uint32_t hi = *cluster.map_shared_rank(&hist_hi[b][tid], c);
                    t += (static_cast<unsigned long long>(hi) << 32) + lo;
                } else {
                    t += *cluster.map_shared_rank(&hist_cnt[b][tid], c);
                }
            }
        return t;
    };
    // From the weights at positions 0..511 (one per thread; position 0 first): the
    // first position where the cumulative weight reaches target or, if that
    // is out of reach, the last position holding any weight.  *above: weight
    // before it; *at: its weight.
    auto pick = [&](unsigned long long tot, unsigned long long target, unsigned long long* above,
                    unsigned long long* at) -> int {
        unsigned long long incl = 0;
        if (tid < kLawBins) {
            incl = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += n;
            }
            if (lane == 31) S.scan_w[warp] = incl;
        }
        if (tid == 0) {
            S.sel_first = INT_MAX;
            S.sel_last = -1;
        }
        __syncthreads();
        if (tid < kLawBins) {
            for (int w = 0; w < warp; ++w) incl += S.scan_w[w];
            if (tot > 0) {
                if (incl >= target) atomicMin(&S.sel_first, tid);
                atomicMax(&S.sel_last, tid);
            }
        }
        __syncthreads();
        const int s = S.sel_first != INT_MAX ? S.sel_first : (S.sel_last > 0 ? S.sel_last : 0);
        if (tid == s) {
            S.sel_above = incl - tot;
            S.sel_at = tot;
        }
        __syncthreads();
        *above = S.sel_above;
        *at = S.sel_at;
        return s;
    };
    // The cut by count (top-k, target k) or by mass (top-p, target ceil(p *
    // total)) among the tokens with key >= lo: the largest key K whose tokens
    // with key >= K weigh at least the target.
    auto find_cut = [&](auto tag, uint32_t lo, unsigned long long target) -> LawCut {
        constexpr bool by_mass = decltype(tag)::value;
        auto weight_of = [&](float x) -> unsigned long long {
            if constexpr (by_mass) return law_mass(law_exp(x, m, inv_t));
            else return 1ull;
        };
        // 1. class weights; bits of this thread's tokens above each class edge
        uint32_t b4 = 0u, b8 = 0u, b16 = 0u, kin = 0u;
        {
            uint32_t h[kLawVals] = {0u, 0u, 0u, 0u}, l[kLawVals] = {0u, 0u, 0u, 0u};
            auto pass = [&](auto has_lo) {
                constexpr bool kHasLo = decltype(has_lo)::value;
#pragma unroll 8
                for (int i = 0; i < kLawChunks; ++i) {
                    const int j = i * kLawThreads + tid;
                    const float x = S.xs[j];  // padding: -inf
                    bool p4, p8, p16;
                    class_add<by_mass, kHasLo>(x, m, inv_t, lo, j < nv, h, l, p4, p8, p16);
                    const uint32_t bit = 1u << i;
                    b4 |= p4 ? bit : 0u;
                    b8 |= p8 ? bit : 0u;
                    b16 |= p16 ? bit : 0u;
                    if (kHasLo) kin |= law_key(x) >= lo ? bit : 0u;
                }
            };
            if (lo) {
                pass(LawTag<true>{});
            } else {
                pass(LawTag<false>{});
                kin = 0xFFFFFFFFu;
            }
            unsigned long long v[kLawVals];
            class_sums<by_mass>(h, l, v);
            cluster_sum(v);
        }
        if (by_mass) {
            target = (unsigned long long)ceil(double(A.top_p) * double(S.tot[0]));
            if (target == 0) target = 1;
        }
        int c = 3;
        unsigned long long base = S.tot[3];
        if (S.tot[1] >= target) {
            c = 0;
            base = 0;
        } else if (S.tot[2] >= target) {
            c = 1;
            base = S.tot[1];
        } else if (S.tot[3] >= target) {
            c = 2;
            base = S.tot[2];
        }
        // this thread's tokens of class c (slots holding a token, key >= lo)
        // the slots of this thread (CH of the mask's bits; class 3 is taken
        // as the complement of the class edges, so the mask must stop there)
        uint32_t valid = CH >= 32 ? 0xFFFFFFFFu : (1u << CH) - 1u;
        if (nv < kLawSlice) {
            valid = 0u;
#pragma unroll
            for (int i = 0; i < kLawChunks; ++i) valid |= i * kLawThreads + tid < nv ? 1u << i : 0u;
        }
        const uint32_t mine = kin & valid & (c == 0 ? b4 : c == 1 ? (b8 & ~b4) : c == 2 ? (b16 & ~b8) : ~b16);

        // 2. fine histogram of class c
        uint32_t fmask = 0;
        int f;
        {
            const int b = hist_begin();
            for (uint32_t bits = mine; bits; bits &= bits - 1) {
                const int i = __ffs(bits) - 1;
                const float x = S.xs[i * kLawThreads + tid];
                hist_put(b, law_fine((x - m) * inv_t, c), by_mass, weight_of(x));
            }
            unsigned long long above = 0, at = 0;
            f = pick(hist_end(b, by_mass), target - base, &above, &at);
            base += above;
        }
        for (uint32_t bits = mine; bits; bits &= bits - 1) {
            const int i = __ffs(bits) - 1;
            if (law_fine((S.xs[i * kLawThreads + tid] - m) * inv_t, c) == f) fmask |= 1u << i;
        }
        const unsigned long long need = target - base;  // weight to take from bin f

        // 3. gather bin f's tokens from the cluster
        if (tid == 0) S.gcount = 0;
        __syncthreads();
        {
            const int n_mine = __popc(fmask);
            int incl = n_mine;  // warp-inclusive count
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += n;
            }
            int base_w = 0;
            if (lane == 31 && incl) base_w = atomicAdd(&S.gcount, incl);
            base_w = __shfl_sync(0xffffffffu, base_w, 31);
            int pos = base_w + incl - n_mine;
            for (uint32_t bits = fmask; bits; bits &= bits - 1, ++pos) {
                const int i = __ffs(bits) - 1;
                if (pos < kGatherCap) {
                    const float x = S.xs[i * kLawThreads + tid];
                    S.glist[pos] = GatherEntry{law_key(x), x};
                }
            }
        }
        __syncthreads();
        cluster.sync();
        if (warp == 0) {
            const int cnt = lane < C ? cluster.map_shared_rank(&S, lane)->gcount : 0;
            int incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += n;
            }
            const bool over = __any_sync(0xffffffffu, cnt > kGatherCap);
            const int total = __shfl_sync(0xffffffffu, incl, 31);  // lanes >= C add nothing
            if (lane < C) S.goff[lane] = incl - cnt;
            if (lane == 0) S.goff[kLawMaxCluster] = over ? INT_MAX : total;
        }
        __syncthreads();
        const int n = S.goff[kLawMaxCluster];
        LawCut cut;
        if (n <= kGatherTotal) {
            // every CTA ranks the n gathered tokens by key
            if (tid < n) {
                int cc = 0;
                while (cc + 1 < C && S.goff[cc + 1] <= tid) ++cc;
                const GatherEntry e = cluster.map_shared_rank(&S, cc)->glist[tid - S.goff[cc]];
                S.gall[tid] = e;
                S.gw[tid] = weight_of(e.x);
            }
            if (tid == 0) {
                S.sel_key = 0u;
                S.sel_min = 0xFFFFFFFFu;
                S.sel_any = 0;
                S.sel_idx = INT_MAX;
            }
            __syncthreads();
            unsigned long long ge = 0, eq = 0;  // weight of the gathered tokens with key >= / == this one
            uint32_t kt = 0;
            if (tid < n) {
                kt = S.gall[tid].key;
                for (int u = 0; u < n; ++u) {
                    const uint32_t ku = S.gall[u].key;
                    const unsigned long long wu = S.gw[u];
                    ge += ku >= kt ? wu : 0ull;
                    eq += ku == kt ? wu : 0ull;
                }
                if (ge >= need) {
                    atomicMax(&S.sel_key, kt);
                    S.sel_any = 1;
                }
                atomicMin(&S.sel_min, kt);
            }
            __syncthreads();
            // out of reach (rounding only): everything in the bin is kept
            const uint32_t K = S.sel_any ? S.sel_key : S.sel_min;
            if (tid < n && kt == K) atomicMin(&S.sel_idx, tid);
            __syncthreads();
            if (tid == S.sel_idx) {
                S.sel_above = ge - eq;
                S.sel_at = eq;
            }
            __syncthreads();
            cut.key = n > 0 ? K : lo;
            cut.above = base + (n > 0 ? S.sel_above : 0ull);
            cut.at = n > 0 ? S.sel_at : 0ull;
        } else {
            // too many to gather: radix select over the keys of bin f
            uint32_t prefix = 0;
            unsigned long long acc = 0, at = 0, tgt = need;
            for (int rr = 0; rr < 4; ++rr) {
                const int shift = 24 - 8 * rr;
                const int b = hist_begin();
                for (uint32_t bits = fmask; bits; bits &= bits - 1) {
                    const int i = __ffs(bits) - 1;
                    const float x = S.xs[i * kLawThreads + tid];
                    const uint32_t k = law_key(x);
                    if (rr > 0 && (k >> (shift + 8)) != prefix) continue;
                    hist_put(b, 255 - int((k >> shift) & 255u), by_mass, weight_of(x));
                }
                unsigned long long a = 0;
                const int s = pick(hist_end(b, by_mass), tgt, &a, &at);
                prefix = (prefix << 8) | uint32_t(255 - s);
                acc += a;
                tgt -= a;
            }
            cut.key = prefix;
            cut.above = base + acc;
            cut.at = at;
        }
        return cut;
    };

    if (st.ok) {
        uint32_t cut = 0;
        unsigned long long kept = 0;
        const bool topk = A.top_k > 0 && A.top_k < V;
        const bool topp = A.top_p < 1.f;
        if (topk) cut = find_cut(LawTag<false>{}, 0u, (unsigned long long)A.top_k).key;
        if (topp) {
            const LawCut c = find_cut(LawTag<true>{}, cut, 0ull);
            cut = c.key;
            kept = c.above + c.at;
        } else {
            // the kept mass, one cluster reduction
            uint32_t hs = 0u, ls = 0u;
#pragma unroll 8
            for (int i = 0; i < kLawChunks; ++i) {
                const float x = S.xs[i * kLawThreads + tid];  // padding: -inf, no mass
                uint32_t hb, lb;
                law_mass_digits(law_key(x) >= cut ? law_exp(x, m, inv_t) : 0.f, hb, lb);
                hs += hb - kMassBias;
                ls += lb - kMassBias;
            }
            unsigned long long v[kLawVals] = {(static_cast<unsigned long long>(hs) << 23) + ls, 0ull, 0ull, 0ull};
            cluster_sum(v);
            kept = S.tot[0];
        }
        st.cut = cut;
        st.inv_s = kept > 0 ? float(70368744177664.0 / double(kept)) : 0.f;
        if (kept == 0) st.ok = 0;
    }
    if (!st.ok && rank == 0 && tid == 0) report(A.status, MXS_DEV_NO_LAW);
    if (A.stats && rank == 0 && tid == 0) A.stats[r] = st;
    if (A.probs) {
        float* out = A.probs + r * V + v0;
#pragma unroll 8
        for (int i = 0; i < kLawChunks; ++i) {
            const int j = i * kLawThreads + tid;
            const float v = law_value(S.xs[j], st, inv_t);
            if (j < nv) out[j] = v;
        }
    }
    cluster.sync();  // no CTA leaves while another may still read its shared memory
}

// ---------------------------------------------------------------------------
// Row form, for batches of many rows: one CTA of 1024 threads per row and no
// cluster.  No row is held on chip: every pass streams the row again (the
// first pass from HBM, the later ones from L2, which holds the rows of all
// CTAs in flight), so about one row per SM is in flight against 36 rows for
// the cluster form, whose slices fill shared memory, and the steps need
// block barriers only.  The steps and every decision are the cluster form's
// (the same classes, fine bins, gather and radix fallback on the same keys
// and fixed-point weights), so both forms give the same statistics bit for
// bit.  (Measured alternatives, 576 rows, top-p: two CTAs of 512 threads per
// SM, 432 us; the row streamed through a shared-memory ring of 1-D bulk
// copies, 489 us; this form, 400 us.  Each pass is bound by instruction issue
// on its SM, not by the bytes in flight.)
// ---------------------------------------------------------------------------
constexpr int kRowThreads = 1024;
constexpr int kRowWarps = kRowThreads / 32;
constexpr int kRowUnroll = 4;  // 16-byte loads in flight per thread in a pass
static_assert(kRowThreads >= kLawBins, "one fine-histogram bin per thread in pick");

// The 16-byte-aligned body of a row (rows are 4-byte aligned): logits
// [head, head + 4 n4) as float4, the rest (at most 3 at each end) scalar.
struct RowSpan {
    int64_t head, n4, tail0;
    __device__ RowSpan(const float* row, int64_t V) {
        head = ((16 - (reinterpret_cast<uintptr_t>(row) & 15)) & 15) >> 2;
        if (head > V) head = V;
        n4 = (V - head) >> 2;
        tail0 = head + (n4 << 2);
    }
};

// f(x) for every logit of the row, each thread a strided share.
template <class F>
__device__ __forceinline__ void row_visit(const float* __restrict__ row, int64_t V, F&& f) {
    const int tid = threadIdx.x;
    const RowSpan s(row, V);
    if (tid < s.head) f(__ldg(row + tid));
    if (tid < V - s.tail0) f(__ldg(row + s.tail0 + tid));
    const float4* body = reinterpret_cast<const float4*>(row + s.head);
    int64_t i = tid;
    for (; i + (kRowUnroll - 1) * kRowThreads < s.n4; i += kRowUnroll * kRowThreads) {
        float4 v[kRowUnroll];
#pragma unroll
        for (int u = 0; u < kRowUnroll; ++u) v[u] = __ldg(body + i + u * kRowThreads);
#pragma unroll
        for (int u = 0; u < kRowUnroll; ++u) {
            f(v[u].x);
            f(v[u].y);
            f(v[u].z);
            f(v[u].w);
        }
    }
    for (; i < s.n4; i += kRowThreads) {
        const float4 v = __ldg(body + i);
        f(v.x);
        f(v.y);
        f(v.z);
        f(v.w);
    }
}

// out[t] = f(row[t]) for every logit of the row (16-byte stores where out
// has the row's alignment phase).
template <class F>
__device__ __forceinline__ void row_map(const float* __restrict__ row, float* __restrict__ out, int64_t V, F&& f) {
    const int tid = threadIdx.x;
    const RowSpan s(row, V);
    if (tid < s.head) out[tid] = f(__ldg(row + tid));
    if (tid < V - s.tail0) out[s.tail0 + tid] = f(__ldg(row + s.tail0 + tid));
    const bool vec = ((reinterpret_cast<uintptr_t>(out) ^ reinterpret_cast<uintptr_t>(row)) & 15) == 0;
    const float4* body = reinterpret_cast<const float4*>(row + s.head);
    float* ob = out + s.head;
    for (int64_t i = tid; i < s.n4; i += kRowThreads) {
        const float4 v = __ldg(body + i);
        const float4 o = make_float4(f(v.x), f(v.y), f(v.z), f(v.w));
        if (vec) {
            *reinterpret_cast<float4*>(ob + 4 * i) = o;
        } else {
            ob[4 * i] = o.x;
            ob[4 * i + 1] = o.y;
            ob[4 * i + 2] = o.z;
            ob[4 * i + 3] = o.w;
        }
    }
}

__global__ void __launch_bounds__(kRowThreads, 1) sampling_law_row_kernel(const LawArgs A) {
    __shared__ uint32_t hist_cnt[kLawBins], hist_lo[kLawBins], hist_hi[kLawBins];
    __shared__ GatherEntry gall[kGatherTotal];
    __shared__ unsigned long long gw[kGatherTotal];
    __shared__ unsigned long long red[kRowWarps][kLawVals];
    __shared__ unsigned long long tot[kLawVals];
    __shared__ unsigned long long scan_w[kLawBins / 32];
    __shared__ unsigned long long sel_above, sel_at;
    __shared__ int gcount, sel_first, sel_last, sel_any, sel_idx;
    __shared__ uint32_t sel_key, sel_min;
    __shared__ float sh_m, sh_tlo, sh_thi;
    __shared__ int sh_bad;

    const int64_t r = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t V = A.V;
    const float* row = r < A.R1 ? A.logits + r * V : A.logits2 + (r - A.R1) * V;

    // ---- the largest finite logit m, and NaN / +inf
    {
        float mx = -INFINITY;
        int bad = 0;
        row_visit(row, V, [&](float v) {
            bad |= int(v != v);
            mx = fmaxf(mx, v);  // NaN ignored; +inf makes the row bad below
        });
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            bad |= __shfl_xor_sync(0xffffffffu, bad, o);
        }
        if (lane == 0) {
            red[warp][0] = __float_as_uint(mx);
            red[warp][1] = unsigned(bad);
        }
        __syncthreads();
        if (tid == 0) {
            float a = -INFINITY;
            int b = 0;
            for (int w = 0; w < kRowWarps; ++w) {
                a = fmaxf(a, __uint_as_float(uint32_t(red[w][0])));
                b |= int(red[w][1]);
            }
            sh_m = a;
            sh_bad = b;
        }
        __syncthreads();
    }
    const float m = sh_m;
    const float inv_t = A.inv_t;
    LawStats st;
    st.m = m;
    st.cut = 0;
    st.inv_s = 0.f;
    st.ok = !sh_bad && m > -INFINITY && m < INFINITY;

    // Sums of kLawVals values over the CTA, into tot (all threads).
    auto block_sum = [&](unsigned long long (&v)[kLawVals]) {
#pragma unroll
        for (int j = 0; j < kLawVals; ++j) v[j] = warp_sum_u64(v[j]);
        if (lane == 0)
#pragma unroll
            for (int j = 0; j < kLawVals; ++j) red[warp][j] = v[j];
        __syncthreads();
        if (tid < kLawVals) {
            unsigned long long t = 0;
            for (int w = 0; w < kRowWarps; ++w) t += red[w][tid];
            tot[tid] = t;
        }
        __syncthreads();
    };
    auto hist_begin = [&]() {
        if (tid < kLawBins) {
            hist_cnt[tid] = 0;
            hist_lo[tid] = 0;
            hist_hi[tid] = 0;
        }
        __syncthreads();
    };
    auto hist_put = [&](int bin, bool by_mass, unsigned long long w) {
        if (!by_mass) {
            atomicAdd(&hist_cnt[bin], 1u);
            return;
        }
        const uint32_t lo = uint32_t(w);
        uint32_t hi = uint32_t(w >> 32);
        const uint32_t old = atomicAdd(&hist_lo[bin], lo);
        if (old + lo < old) ++hi;
        if (hi) atomicAdd(&hist_hi[bin], hi);
    };
    // After the pass: the weight at bin tid (threads below kLawBins).
    auto hist_end = [&](bool by_mass) -> unsigned long long {
        __syncthreads();
        if (tid >= kLawBins) return 0ull;
        return by_mass ? (static_cast<unsigned long long>(hist_hi[tid]) << 32) + hist_lo[tid]
                       : static_cast<unsigned long long>(hist_cnt[tid]);
    };
    // As the cluster form's pick: the first of 512 positions where the
    // cumulative weight reaches target, else the last one holding weight.
    auto pick = [&](unsigned long long w, unsigned long long target, unsigned long long* above,
                    unsigned long long* at) -> int {
        unsigned long long incl = 0;
        if (tid < kLawBins) {
            incl = w;
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
        if (tid < kLawBins) {
            for (int q = 0; q < warp; ++q) incl += scan_w[q];
            if (w > 0) {
                if (incl >= target) atomicMin(&sel_first, tid);
                atomicMax(&sel_last, tid);
            }
        }
        __syncthreads();
        const int s = sel_first != INT_MAX ? sel_first : (sel_last > 0 ? sel_last : 0);
        if (tid == s) {
            sel_above = incl - w;
            sel_at = w;
        }
        __syncthreads();
        *above = sel_above;
        *at = sel_at;
        return s;
    };

    // The cut by count or by mass among the tokens with key >= lo (the
    // cluster form's find_cut, streaming the row for each step).
    auto find_cut = [&](auto tag, uint32_t lo, unsigned long long target) -> LawCut {
        constexpr bool by_mass = decltype(tag)::value;
        auto weight_of = [&](float x) -> unsigned long long {
            if constexpr (by_mass) return law_mass(law_exp(x, m, inv_t));
            else return 1ull;
        };
        // 1. class weights
        {
            uint32_t h[kLawVals] = {0u, 0u, 0u, 0u}, l[kLawVals] = {0u, 0u, 0u, 0u};
            auto pass = [&](auto has_lo) {
                row_visit(row, V, [&](float x) {
                    bool p4, p8, p16;
                    class_add<by_mass, decltype(has_lo)::value>(x, m, inv_t, lo, true, h, l, p4, p8, p16);
                });
            };
            if (lo) pass(LawTag<true>{});
            else pass(LawTag<false>{});
            unsigned long long v[kLawVals];
            class_sums<by_mass>(h, l, v);
            block_sum(v);
        }
        if (by_mass) {
            target = (unsigned long long)ceil(double(A.top_p) * double(tot[0]));
            if (target == 0) target = 1;
        }
        int c = 3;
        unsigned long long base = tot[3];
        if (tot[1] >= target) {
            c = 0;
            base = 0;
        } else if (tot[2] >= target) {
            c = 1;
            base = tot[1];
        } else if (tot[3] >= target) {
            c = 2;
            base = tot[2];
        }
        __syncthreads();  // tot is read by all before the next block_sum

        // 2. fine histogram of class c
        int f;
        {
            hist_begin();
            auto fine_pass = [&](auto has_lo) {
                row_visit(row, V, [&](float x) {
                    const float a = (x - m) * inv_t;
                    if (in_class(a, c) && (!decltype(has_lo)::value || law_key(x) >= lo))
                        hist_put(law_fine(a, c), by_mass, weight_of(x));
                });
            };
            if (lo) fine_pass(LawTag<true>{});
            else fine_pass(LawTag<false>{});
            unsigned long long above = 0, at = 0;
            f = pick(hist_end(by_mass), target - base, &above, &at);
            base += above;
        }
        const unsigned long long need = target - base;

        // 3. gather bin f's tokens (bin f as an interval of t = -a)
        if (tid == 0) {
            gcount = 0;
            fine_bin_range(c, f, &sh_tlo, &sh_thi);
        }
        __syncthreads();
        {
            const float tlo = sh_tlo, thi = sh_thi;
            auto gather_pass = [&](auto has_lo) {
                row_visit(row, V, [&](float x) {
                    const float a = (x - m) * inv_t;
                    if (in_class(a, c) && -a >= tlo && -a <= thi &&
                        (!decltype(has_lo)::value || law_key(x) >= lo)) {
                        const int pos = atomicAdd(&gcount, 1);
                        if (pos < kGatherTotal) gall[pos] = GatherEntry{law_key(x), x};
                    }
                });
            };
            if (lo) gather_pass(LawTag<true>{});
            else gather_pass(LawTag<false>{});
        }
        __syncthreads();
        const int n = gcount;
        LawCut cut;
        if (n <= kGatherTotal) {
            if (tid < n) gw[tid] = weight_of(gall[tid].x);
            if (tid == 0) {
                sel_key = 0u;
                sel_min = 0xFFFFFFFFu;
                sel_any = 0;
                sel_idx = INT_MAX;
            }
            __syncthreads();
            unsigned long long ge = 0, eq = 0;
            uint32_t kt = 0;
            if (tid < n) {
                kt = gall[tid].key;
                for (int u = 0; u < n; ++u) {
                    const uint32_t ku = gall[u].key;
                    const unsigned long long wu = gw[u];
                    ge += ku >= kt ? wu : 0ull;
                    eq += ku == kt ? wu : 0ull;
                }
                if (ge >= need) {
                    atomicMax(&sel_key, kt);
                    sel_any = 1;
                }
                atomicMin(&sel_min, kt);
            }
            __syncthreads();
            const uint32_t K = sel_any ? sel_key : sel_min;
            if (tid < n && kt == K) atomicMin(&sel_idx, tid);
            __syncthreads();
            if (tid == sel_idx) {
                sel_above = ge - eq;
                sel_at = eq;
            }
            __syncthreads();
            cut.key = n > 0 ? K : lo;
            cut.above = base + (n > 0 ? sel_above : 0ull);
            cut.at = n > 0 ? sel_at : 0ull;
            __syncthreads();  // sel_* are reused by the next step
        } else {
            // too many to gather: radix select over the keys of bin f
            uint32_t prefix = 0;
            unsigned long long acc = 0, at = 0, tgt = need;
            for (int rr = 0; rr < 4; ++rr) {
                const int shift = 24 - 8 * rr;
                hist_begin();
                row_visit(row, V, [&](float x) {
                    const float a = (x - m) * inv_t;
                    const uint32_t k = law_key(x);
                    if (!in_class(a, c) || k < lo || law_fine(a, c) != f) return;
                    if (rr > 0 && (k >> (shift + 8)) != prefix) return;
                    hist_put(255 - int((k >> shift) & 255u), by_mass, weight_of(x));
                });
                unsigned long long a = 0;
                const int s = pick(hist_end(by_mass), tgt, &a, &at);
                prefix = (prefix << 8) | uint32_t(255 - s);
                acc += a;
                tgt -= a;
            }
            cut.key = prefix;
            cut.above = base + acc;
            cut.at = at;
        }
        return cut;
    };

    if (st.ok) {
        uint32_t cut = 0;
        unsigned long long kept = 0;
        const bool topk = A.top_k > 0 && A.top_k < V;
        const bool topp = A.top_p < 1.f;
        if (topk) cut = find_cut(LawTag<false>{}, 0u, (unsigned long long)A.top_k).key;
        if (topp) {
            const LawCut c = find_cut(LawTag<true>{}, cut, 0ull);
            cut = c.key;
            kept = c.above + c.at;
        } else {
            uint32_t hs = 0u, ls = 0u;
            row_visit(row, V, [&](float x) {
                uint32_t hb, lb;
                law_mass_digits(law_key(x) >= cut ? law_exp(x, m, inv_t) : 0.f, hb, lb);
                hs += hb - kMassBias;
                ls += lb - kMassBias;
            });
            unsigned long long v[kLawVals] = {(static_cast<unsigned long long>(hs) << 23) + ls, 0ull, 0ull, 0ull};
            block_sum(v);
            kept = tot[0];
        }
        st.cut = cut;
        st.inv_s = kept > 0 ? float(70368744177664.0 / double(kept)) : 0.f;
        if (kept == 0) st.ok = 0;
    }
    if (!st.ok && tid == 0) report(A.status, MXS_DEV_NO_LAW);
    if (A.stats && tid == 0) A.stats[r] = st;
    if (A.probs) row_map(row, A.probs + r * V, V, [&](float x) { return law_value(x, st, inv_t); });
}

// The form for R rows (MXS_LAW_FORM=cluster16 / cluster / row overrides).
// Measured at V = 128256, top-p: 80 rows 71 us (clusters of 8) / 99 us (row);
// 144 rows 124 / 112 us; 576 rows 433 / 400 us.  Below ~100 rows the cluster
// form spreads each row over 4 SMs; above, the row form keeps more rows in
// flight.  When clusters of 8 would leave most SMs idle (R * C <= 76), the
// narrow slices (8192 logits, clusters of up to 16) spread each row over
// twice the SMs: 1 row 18.7 / 10.5 us (top-p / plain) against 20.7 / 14.4;
// 4 rows 20.6 / 10.4 against 20.6 / 14.4; even at 9 rows; slower from 16.
constexpr int64_t kLawRowMinRows = 128;
enum class LawForm { kNarrow, kWide, kRow };
static LawForm law_form(int64_t R, int64_t V) {
    if (const char* f = std::getenv("MXS_LAW_FORM")) {
        if (std::strcmp(f, "row") == 0) return LawForm::kRow;
        if (std::strcmp(f, "cluster") == 0) return LawForm::kWide;
        if (std::strcmp(f, "cluster16") == 0) return LawForm::kNarrow;
    }
    if (R >= kLawRowMinRows) return LawForm::kRow;
    const int64_t c8 = (V + int64_t(kLawThreads) * kLawChunksWide - 1) / (int64_t(kLawThreads) * kLawChunksWide);
    return R * c8 <= 76 ? LawForm::kNarrow : LawForm::kWide;
}

// One cluster of C = ceil(V / (512 CH)) CTAs per row.
template <int CH>
static cudaError_t launch_law_cluster(const LawArgs& A, cudaStream_t stream) {
    constexpr int64_t kSlice = int64_t(kLawThreads) * CH;
    constexpr int kSmem = int(sizeof(LawSmem<CH>));
    const int C = int((A.V + kSlice - 1) / kSlice);
    static const cudaError_t attr_err = [] {
        cudaError_t e = cudaFuncSetAttribute(sampling_law_kernel<CH>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (e == cudaSuccess && law_max_cluster<CH>() > 8)  // clusters beyond the portable 8
            e = cudaFuncSetAttribute(sampling_law_kernel<CH>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        return e;
    }();
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(unsigned(A.R * C), 1, 1);
    cfg.blockDim = dim3(kLawThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = unsigned(C);
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, sampling_law_kernel<CH>, A);
}

static cudaError_t launch_law(const LawArgs& A, cudaStream_t stream) {
    if (A.R < 1) return cudaSuccess;
    switch (law_form(A.R, A.V)) {
        case LawForm::kRow:
            sampling_law_row_kernel<<<unsigned(A.R), kRowThreads, 0, stream>>>(A);
            return cudaGetLastError();
        case LawForm::kNarrow:
            return launch_law_cluster<kLawChunksNarrow>(A, stream);
        default:
            return launch_law_cluster<kLawChunksWide>(A, stream);
    }
}

static LawArgs law_args(const float* logits, int64_t R, int64_t V, const LawSampling& s, int32_t* status) {
    LawArgs A{};
    A.logits = logits;
    A.logits2 = nullptr;
    A.R1 = R;
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

cudaError_t law_stats_run2(const float* logits_a, int64_t Ra, const float* logits_b, int64_t Rb, int64_t V,
                           const LawSampling& s, LawStats* stats, int32_t* dev_status, cudaStream_t stream) {
    LawArgs A = law_args(logits_a, Ra + Rb, V, s, dev_status);
    A.logits2 = logits_b;
    A.R1 = Ra;
    A.stats = stats;
    return launch_law(A, stream);
}

}  // namespace mxs
