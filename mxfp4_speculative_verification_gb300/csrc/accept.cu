// spec_accept on sm_103a: exact left-to-right acceptance, residual or bonus
// sampling and emission of 1..K+1 tokens per sequence.
//
// Operation: "Module 11. Speculative Decoding and Quantization", §4 (accept
// x_i with probability min(1, p_i(x_i)/q_i(x_i)) from left to right; at the
// first rejection draw the replacement from norm((p - q)+); when every
// proposal survives draw the bonus token from the next position's law) and
// §5 (block B18: the draw is accepted iff draw < acceptance, acceptance 0
// where q = 0).  The pipeline diagram of "Next-Gen Speculative Decoding and
// FP4 Quantization Shake Up LLM Inference Economics" names this step the
// "Parallel Softmax & Acceptance Evaluation Mask" of the batched
// verification kernel.
//
// Two kernels.  For V <= 131072 (the pages' vocabularies) the register-
// resident kernel further down holds each CTA's slice of the sampled law in
// registers and carries the CDF in float-float arithmetic.  Above that, the
// streaming kernel below: one thread-block cluster of C CTAs per sequence
// (C = 1..8 by vocabulary size), each CTA owning a contiguous slice of the
// vocabulary:
//  * warp 0 of every CTA gathers p_i(x_i), q_i(x_i), u_i for the K drafts,
//    tests u*q < p exactly (an fp32 x fp32 product is exact in double) and
//    finds the first rejection j with one ballot (all CTAs agree);
//  * all warps stream their slice of the one law that is sampled (residual
//    row pair j, or p_K) with float4 loads, forming fp32 sums of 128-element
//    sub-tiles in shared memory and the slice total in double;
//  * the slice totals are exchanged through distributed shared memory and
//    summed in rank order by every CTA (identical S everywhere); the CTA
//    whose slice holds the crossing C_t > u_K * S locates the sub-tile with a
//    double scan and rescans it in double to pick the token.
#include <cooperative_groups.h>

#include <atomic>
#include <climits>
#include <cstdlib>

#include "law.cuh"
#include "mxs_device.cuh"
#include "mxs_internal.h"

namespace cg = cooperative_groups;

namespace mxs {

constexpr int kAcceptThreads = 512;
constexpr int kAcceptWarps = kAcceptThreads / 32;
constexpr int kSubTile = 128;  // elements per warp step (float4 per lane)
constexpr int kMaxCluster = 8;
constexpr double kNearEdge = 1e-5;

struct AcceptParams {
    const float* p;
    const float* q;
    const int32_t* draft;
    const float* u;
    int64_t V;
    int K;
    int nsub;       // ceil(V / kSubTile)
    int per_cta;    // sub-tiles per CTA of the cluster
    int32_t* out_tokens;
    int32_t* n_emitted;
    int32_t* row_flags;
    int32_t* status;
    // laws given as logits (p and q then point at logit rows): each row's
    // statistics, and 1 / temperature; p_t = law_value(logit_t, stats, inv_t)
    const LawStats* pst;  // [B, K+1]
    const LawStats* qst;  // [B, K]
    float inv_t;
};

// What each CTA publishes to the others of its cluster.
struct SliceSummary {
    double total;  // sum of the slice's sub-tile sums (double, fixed order)
    int lastpos;   // last index with positive mass in the slice (-1 if none)
};

// Residual (or bonus) mass of 4 consecutive elements starting at e.
template <bool VEC>
__device__ __forceinline__ void load_law4(const float* __restrict__ prow,
                                          const float* __restrict__ qrow, bool use_res, int64_t e,
                                          int64_t V, float (&r)[4]) {
    if (VEC && e + 3 < V) {
        const float4 pv = __ldcs(reinterpret_cast<const float4*>(prow + e));
        if (use_res) {
            const float4 qv = __ldcs(reinterpret_cast<const float4*>(qrow + e));
            r[0] = fmaxf(pv.x - qv.x, 0.f);
            r[1] = fmaxf(pv.y - qv.y, 0.f);
            r[2] = fmaxf(pv.z - qv.z, 0.f);
            r[3] = fmaxf(pv.w - qv.w, 0.f);
        } else {
            r[0] = pv.x; r[1] = pv.y; r[2] = pv.z; r[3] = pv.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float v = 0.f;
            if (e + i < V) {
                const float pv = prow[e + i];
                v = use_res ? fmaxf(pv - qrow[e + i], 0.f) : pv;
            }
            r[i] = v;
        }
    }
}

// The same for laws given as logits with their row statistics (LG), or as
// probabilities (then the same as load_law4).
template <bool VEC, bool LG>
__device__ __forceinline__ void load_law4x(const float* __restrict__ prow, const float* __restrict__ qrow,
                                           bool use_res, int64_t e, int64_t V, float (&r)[4],
                                           const LawStats& ps, const LawStats& qs, float inv_t) {
    if constexpr (!LG) {
        load_law4<VEC>(prow, qrow, use_res, e, V, r);
    } else {
        float pl[4], ql[4];
        if (VEC && e + 3 < V) {
            const float4 pv = __ldcs(reinterpret_cast<const float4*>(prow + e));
            pl[0] = pv.x; pl[1] = pv.y; pl[2] = pv.z; pl[3] = pv.w;
            if (use_res) {
                const float4 qv = __ldcs(reinterpret_cast<const float4*>(qrow + e));
                ql[0] = qv.x; ql[1] = qv.y; ql[2] = qv.z; ql[3] = qv.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                pl[i] = e + i < V ? prow[e + i] : -INFINITY;
                ql[i] = (use_res && e + i < V) ? qrow[e + i] : -INFINITY;
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float v = 0.f;
            if (e + i < V) {
                const float pv = law_value(pl[i], ps, inv_t);
                v = use_res ? fmaxf(pv - law_value(ql[i], qs, inv_t), 0.f) : pv;
            }
            r[i] = v;
        }
    }
}

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Inclusive warp scan (double).
__device__ __forceinline__ double warp_scan_d(double v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

// Stream sub-tiles [s0, s1) of the law once: fp32 sums into subsum[st - s0],
// the last positive index into *lastpos.
template <bool VEC>
__device__ void sum_pass(const float* __restrict__ prow, const float* __restrict__ qrow,
                         bool use_res, int64_t V, int s0, int s1, float* subsum, int* lastpos) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int lp = -1;
    constexpr int U = 4;
    for (int st0 = s0 + warp; st0 < s1; st0 += U * kAcceptWarps) {
        float r[U][4];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int st = st0 + k * kAcceptWarps;
            if (st < s1) {
                load_law4<VEC>(prow, qrow, use_res, int64_t(st) * kSubTile + 4 * lane, V, r[k]);
            } else {
                r[k][0] = r[k][1] = r[k][2] = r[k][3] = 0.f;
            }
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int st = st0 + k * kAcceptWarps;
            if (st >= s1) break;
            const float s = warp_sum_f((r[k][0] + r[k][1]) + (r[k][2] + r[k][3]));
            if (lane == 0) subsum[st - s0] = s;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (r[k][i] > 0.f) lp = max(lp, st * kSubTile + 4 * lane + i);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, o));
    if (lane == 0 && lp >= 0) atomicMax(lastpos, lp);
}

// Sum of the slice's sub-tile sums in a fixed order (thread-strided, then tree).
__device__ double slice_total(const float* subsum, int n, double* wtot) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    double s = 0.0;
    for (int i = threadIdx.x; i < n; i += kAcceptThreads) s += double(subsum[i]);
    s = warp_sum_d(s);
    if (lane == 0) wtot[warp] = s;
    __syncthreads();
    double S = 0.0;
    for (int w = 0; w < kAcceptWarps; ++w) S += wtot[w];
    __syncthreads();
    return S;
}

// The left-to-right acceptance test of row b, run by one warp: lane i < K
// gathers p_i(x_i), q_i(x_i) and u_i, tests u*q < p exactly (an fp32 x fp32
// product is exact in double) and one ballot finds the first rejection j (K if
// every draft survives).  Lane 0 stores j and the row's flags.
template <bool LG = false>
__device__ __forceinline__ void accept_drafts(const AcceptParams& P, int64_t b, int lane, int* sh_j,
                                              int* sh_flags, int* sh_err) {
    const int K = P.K;
    const int64_t V = P.V;
    const bool active = lane < K;
    const int x = active ? P.draft[b * K + lane] : 0;
    const bool bad = active && (x < 0 || int64_t(x) >= V);
    const unsigned badm = __ballot_sync(0xffffffffu, bad);
    int j = K, flags = 0;
    if (badm) {
        flags = MXS_DEV_BAD_DRAFT;
    } else {
        bool rej = false, zq = false;
        if (active) {
            float qx = P.q[(b * K + lane) * V + x];
            float px = P.p[(b * (K + 1) + lane) * V + x];
            if constexpr (LG) {
                qx = law_value(qx, P.qst[b * K + lane], P.inv_t);
                px = law_value(px, P.pst[b * (K + 1) + lane], P.inv_t);
            }
            const float ui = P.u[b * (K + 1) + lane];
            if (qx > 0.f) {
                rej = !(double(ui) * double(qx) < double(px));
            } else {
                rej = true;
                zq = true;
            }
        }
        const unsigned rm = __ballot_sync(0xffffffffu, rej);
        const unsigned zm = __ballot_sync(0xffffffffu, zq);
        if (rm) {
            j = __ffs(int(rm)) - 1;
            if ((zm >> j) & 1u) flags |= MXS_DEV_ZERO_Q;
        }
    }
    if (lane == 0) {
        *sh_j = j;
        *sh_flags = flags;
        *sh_err = badm ? 1 : 0;
    }
}

template <bool VEC>
__global__ void __launch_bounds__(kAcceptThreads) spec_accept_kernel(const AcceptParams P) {
    extern __shared__ float subsum[];
    __shared__ double wtot[kAcceptWarps];
    __shared__ double sh_prefix;
    __shared__ SliceSummary sh_mine;
    __shared__ int sh_j, sh_flags, sh_err, sh_lastpos, sh_tstar;

    cg::cluster_group cluster = cg::this_cluster();
    const int C = int(cluster.num_blocks());
    const int rank = int(cluster.block_rank());
    const int64_t b = blockIdx.x / C;
    const int K = P.K;
    const int64_t V = P.V;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---------------------------------------------- acceptance (warp 0)
    if (warp == 0) {
        accept_drafts(P, b, lane, &sh_j, &sh_flags, &sh_err);
        if (lane == 0) {
            sh_lastpos = -1;
            sh_tstar = INT_MAX;
        }
    }
    __syncthreads();

    const int j = sh_j;
    int32_t* tok = P.out_tokens + b * (K + 1);
    if (sh_err) {  // uniform across the cluster: no cluster barrier is reached
        if (rank == 0) {
            for (int i = threadIdx.x; i <= K; i += blockDim.x) tok[i] = -1;
            if (threadIdx.x == 0) {
                P.n_emitted[b] = 0;
                if (P.row_flags) P.row_flags[b] = sh_flags;
                report(P.status, sh_flags);
            }
        }
        return;
    }

    // --------------------------------------- the law: residual or bonus
    bool use_res = j < K;
    const float* prow = P.p + (b * (K + 1) + j) * V;
    const float* qrow = use_res ? P.q + (b * K + j) * V : nullptr;
    const int s0 = min(P.nsub, rank * P.per_cta);
    const int s1 = min(P.nsub, s0 + P.per_cta);
    const int nloc = s1 - s0;

    // Sum this CTA's slice, publish it, and read every slice of the cluster.
    // Returns S (identical bits in every CTA) and this slice's prefix.
    auto exchange = [&](double& S, double& prefix, int& lastpos) {
        sum_pass<VEC>(prow, qrow, use_res, V, s0, s1, subsum, &sh_lastpos);
        __syncthreads();
        const double tot = slice_total(subsum, nloc, wtot);
        if (threadIdx.x == 0) {
            sh_mine.total = tot;
            sh_mine.lastpos = sh_lastpos;
        }
        cluster.sync();
        S = 0.0;
        prefix = 0.0;
        lastpos = -1;
        for (int c = 0; c < C; ++c) {
            const SliceSummary o = *cluster.map_shared_rank(&sh_mine, c);
            if (c == rank) prefix = S;
            S += o.total;
            lastpos = max(lastpos, o.lastpos);
        }
        cluster.sync();  // every CTA has read every summary
    };
    double S, prefix;
    int lastpos;
    exchange(S, prefix, lastpos);
    if (!(S > 0.0)) {
        // A positive residual exists whenever rejection is possible; only the
        // rounding of the inputs gets here.  Sample p_j instead.
        if (threadIdx.x == 0) {
            sh_flags |= MXS_DEV_ZERO_RESIDUAL;
            sh_lastpos = -1;
        }
        __syncthreads();
        use_res = false;
        qrow = nullptr;
        exchange(S, prefix, lastpos);
    }
    const bool no_law = !(S > 0.0) || isinf(S) || isnan(S);
    const double uK = double(P.u[b * (K + 1) + K]);
    const double thr = uK * S;

    // The slice holding the first crossing, computed identically everywhere.
    int owner = -1;
    if (!no_law) {
        double run = 0.0;
        for (int c = 0; c < C; ++c) {
            const double t = cluster.map_shared_rank(&sh_mine, c)->total;
            if (t > 0.0 && run + t > thr) {
                owner = c;
                break;
            }
            run += t;
        }
    }
    // Summaries stay readable until every CTA has located the owner.
    cluster.sync();
    const int writer = (no_law || owner < 0) ? 0 : owner;
    if (rank != writer) return;

    if (no_law) {
        for (int i = threadIdx.x; i <= K; i += blockDim.x) tok[i] = -1;
        if (threadIdx.x == 0) {
            const int f = sh_flags | MXS_DEV_NO_LAW;
            P.n_emitted[b] = 0;
            if (P.row_flags) P.row_flags[b] = f;
            report(P.status, f);
        }
        return;
    }

    // --------------------------- locate the sub-tile where C crosses thr
    if (owner >= 0) {
        const int per = (nloc + kAcceptThreads - 1) / kAcceptThreads;
        const int a0 = min(nloc, int(threadIdx.x) * per);
        const int a1 = min(nloc, a0 + per);
        double local = 0.0;
        for (int st = a0; st < a1; ++st) local += double(subsum[st]);
        const double inc = warp_scan_d(local, lane);
        if (lane == 31) wtot[warp] = inc;
        __syncthreads();
        if (warp == 0) {
            const double wt = lane < kAcceptWarps ? wtot[lane] : 0.0;
            const double winc = warp_scan_d(wt, lane);
            if (lane < kAcceptWarps) wtot[lane] = winc - wt;  // exclusive prefix of warp totals
        }
        __syncthreads();
        double run = prefix + wtot[warp] + (inc - local);
        for (int st = a0; st < a1; ++st) {
            const float s = subsum[st];
            const double end = run + double(s);
            if (s > 0.f && end > thr) {
                atomicMin(&sh_tstar, st);
                break;
            }
            run = end;
        }
        __syncthreads();
        // the owner of the first crossing publishes its starting prefix
        run = prefix + wtot[warp] + (inc - local);
        for (int st = a0; st < a1; ++st) {
            if (st == sh_tstar) sh_prefix = run;
            run += double(subsum[st]);
        }
        __syncthreads();
        if (sh_tstar == INT_MAX && threadIdx.x == 0) {
            // Summed in this order the slice ends at or below u*S (a rounding
            // tie with its total): continue the rescan after the slice.
            double end = prefix;
            for (int st = 0; st < nloc; ++st) end += double(subsum[st]);
            sh_prefix = end;
            sh_tstar = nloc;
        }
        __syncthreads();
    }

    // ------------------------------ warp 0: exact position in the sub-tile
    if (warp == 0) {
        int pick = -1;
        double before = 0.0, after = 0.0;
        if (owner >= 0 && sh_tstar != INT_MAX) {
            double run = sh_prefix;
            for (int st = s0 + sh_tstar; st < P.nsub && pick < 0; ++st) {
                float r[4];
                load_law4<VEC>(prow, qrow, use_res, int64_t(st) * kSubTile + 4 * lane, V, r);
                double c[4];
                c[0] = double(r[0]);
                c[1] = c[0] + double(r[1]);
                c[2] = c[1] + double(r[2]);
                c[3] = c[2] + double(r[3]);
                const double lane_inc = warp_scan_d(c[3], lane);
                const double base = run + (lane_inc - c[3]);
                int first = 4;
#pragma unroll
                for (int i = 3; i >= 0; --i)
                    if (r[i] > 0.f && base + c[i] > thr) first = i;
                const unsigned hit = __ballot_sync(0xffffffffu, first < 4);
                if (hit) {
                    const int L = __ffs(int(hit)) - 1;
                    const int fi = __shfl_sync(0xffffffffu, first, L);
                    const double cb = __shfl_sync(0xffffffffu, base, L);
                    double ci = 0.0, ri = 0.0;
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (i == fi) { ci = c[i]; ri = double(r[i]); }
                    ci = __shfl_sync(0xffffffffu, ci, L);
                    ri = __shfl_sync(0xffffffffu, ri, L);
                    pick = st * kSubTile + 4 * L + fi;
                    after = cb + ci;
                    before = after - ri;
                }
                run += __shfl_sync(0xffffffffu, lane_inc, 31);
            }
        }
        if (pick < 0) {
            // rounding put u*S at or beyond the last positive mass
            pick = lastpos;
            float rl[4];
            const int64_t e = int64_t(pick) & ~int64_t(3);
            load_law4<false>(prow, qrow, use_res, e, V, rl);
            after = S;
            before = S - double(rl[pick - e]);
        }
        if (lane == 0) {
            int flags = sh_flags;
            const double d0 = fabs(uK - before / S), d1 = fabs(uK - after / S);
            if (fmin(d0, d1) < kNearEdge) flags |= MXS_DEV_NEAR_EDGE;
            tok[j] = pick;
            P.n_emitted[b] = j + 1;
            if (P.row_flags) P.row_flags[b] = flags;
            report(P.status, flags);
        }
    }
    // emitted drafts, then padding
    for (int i = threadIdx.x; i <= K; i += blockDim.x) {
        if (i < j) tok[i] = P.draft[b * K + i];
        else if (i > j) tok[i] = -1;
    }
}

// ---------------------------------------------------------------------------
// Register-resident variant for V <= kRegMaxV (every vocabulary of the pages'
// models).  CTA `rank` of the cluster owns elements [rank * 16384, ...) and
// loads them once, 8 float4 per thread with every load in flight; element
// v0 + 4 (i * 512 + t) + e sits in chunk i of thread t, so chunk i of warp w
// is the 128-element sub-tile i * 16 + w and its fp32 sum is formed exactly
// as in the streaming kernel.  After one exchange of slice totals (two
// cluster barriers) the CTA holding the crossing locates the sub-tile and the
// warp that loaded it rescans it from its registers.
//
// Above the sub-tile sums the running CDF is carried in float-float (an fp32
// pair added with error-free transformations, about 44 significant bits):
// dependent double additions cost hundreds of cycles each on this GPU's
// FP64 unit and dominated the latency of a call; the pair arithmetic runs on
// the fp32 pipes and keeps the CDF error many orders below the 1e-5 band in
// which a sampled token may legitimately differ from the oracle's.
// ---------------------------------------------------------------------------
struct ff {
    float hi, lo;
};
__device__ __forceinline__ ff ff_make(float a) { return ff{a, 0.f}; }
// Knuth's two-sum of the high parts, then the low parts folded in.
__device__ __forceinline__ ff ff_add(ff a, ff b) {
    const float s = __fadd_rn(a.hi, b.hi);
    const float v = __fsub_rn(s, a.hi);
    float e = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, v)), __fsub_rn(b.hi, v));
    e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
    const float hi = __fadd_rn(s, e);
    return ff{hi, __fsub_rn(e, __fsub_rn(hi, s))};
}
__device__ __forceinline__ ff ff_neg(ff a) { return ff{-a.hi, -a.lo}; }
// sign of a - b (compared through the pair difference)
__device__ __forceinline__ bool ff_gt(ff a, ff b) {
    const ff d = ff_add(a, ff_neg(b));
    return d.hi > 0.f || (d.hi == 0.f && d.lo > 0.f);
}
// u * a for an fp32 u: the product of the high parts split exactly by an fma
__device__ __forceinline__ ff ff_mul_f(ff a, float u) {
    const float p = __fmul_rn(a.hi, u);
    const float e = __fmaf_rn(a.hi, u, -p);
    return ff_add(ff{p, 0.f}, ff{e, __fmul_rn(a.lo, u)});
}
__device__ __forceinline__ ff ff_shfl_up(ff v, int o) {
    return ff{__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
}
__device__ __forceinline__ ff ff_shfl(ff v, int src) {
    return ff{__shfl_sync(0xffffffffu, v.hi, src), __shfl_sync(0xffffffffu, v.lo, src)};
}
__device__ __forceinline__ ff ff_shfl_xor(ff v, int o) {
    return ff{__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
}
// inclusive warp scan in lane order
__device__ __forceinline__ ff warp_scan_ff(ff v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const ff n = ff_shfl_up(v, o);
        if (lane >= o) v = ff_add(n, v);
    }
    return v;
}
// exclusive prefix from an inclusive scan (lane 0 gets zero)
__device__ __forceinline__ ff warp_excl_ff(ff inc, int lane) {
    const ff e = ff_shfl_up(inc, 1);
    return lane == 0 ? ff{0.f, 0.f} : e;
}

struct SliceSummaryFF {
    ff total;
    int lastpos;
};

constexpr int64_t kRegMaxV = int64_t(kMaxCluster) * kAcceptThreads * 4 * 8;  // 131072

// RELOAD = false keeps the slice in registers until the rescan (one CTA per SM,
// CH = 8 float4 chunks per thread: 16384-element slices; best while every row's
// cluster is resident at once).  RELOAD = true lets the registers go after the
// sub-tile sums (formed in batches of 4 chunks) and re-reads the one crossing
// sub-tile from L2 for the rescan: two CTAs share an SM, and with CH = 16
// (32768-element slices, clusters of 4 at V = 128256) four times as many rows
// are in flight when a batch would otherwise need several waves.
//
// LG = true: the laws are given as logits with per-row statistics (law.cu),
// and every probability is formed on the fly from them: the rows of
// probabilities are never written.
// Reload forms ask for two CTAs per SM, except when each value is formed from
// a logit: the law's temporaries then spilled at that budget.
template <bool VEC, bool RELOAD, int CH, bool LG = false>
__global__ void __launch_bounds__(kAcceptThreads, RELOAD && !LG ? 2 : 1)
    spec_accept_reg_kernel(const AcceptParams P) {
    constexpr int kRegChunks = CH;
    constexpr int kRegSlice = kAcceptThreads * 4 * kRegChunks;  // elements per CTA
    constexpr int kRegSub = kRegChunks * kAcceptWarps;           // 128-element sub-tiles per CTA
    static_assert(kRegSub <= kAcceptThreads, "one sub-tile per thread in the scan");
    __shared__ float subsum[kRegSub];
    __shared__ ff wsum[kRegSub / 32];
    // every CTA's slice summary, written into every CTA of the cluster before
    // one cluster barrier (one buffer per exchange: a second exchange follows
    // when the residual has no mass)
    __shared__ SliceSummaryFF sh_sums[2][kMaxCluster];
    __shared__ ff sh_S, sh_slice_prefix, sh_prefix;
    __shared__ int sh_j, sh_flags, sh_err, sh_lastpos, sh_all_lastpos, sh_owner, sh_tstar;

    cg::cluster_group cluster = cg::this_cluster();
    const int C = int(cluster.num_blocks());
    const int rank = int(cluster.block_rank());
    const int64_t b = blockIdx.x / C;
    const int K = P.K;
    const int64_t V = P.V;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == 0) {
        accept_drafts<LG>(P, b, lane, &sh_j, &sh_flags, &sh_err);
        if (lane == 0) sh_tstar = INT_MAX;
    }
    __syncthreads();

    const int j = sh_j;
    int32_t* tok = P.out_tokens + b * (K + 1);
    if (sh_err) {  // uniform across the cluster: no cluster barrier is reached
        if (rank == 0) {
            for (int i = threadIdx.x; i <= K; i += blockDim.x) tok[i] = -1;
            if (threadIdx.x == 0) {
                P.n_emitted[b] = 0;
                if (P.row_flags) P.row_flags[b] = sh_flags;
                report(P.status, sh_flags);
            }
        }
        return;
    }

    bool use_res = j < K;
    const float* prow = P.p + (b * (K + 1) + j) * V;
    const float* qrow = use_res ? P.q + (b * K + j) * V : nullptr;
    const int64_t v0 = int64_t(rank) * kRegSlice;
    const float uK = P.u[b * (K + 1) + K];
    float r[kRegChunks][4];
    LawStats ps{}, qs{};
    if constexpr (LG) {
        ps = P.pst[b * (K + 1) + j];
        if (use_res) qs = P.qst[b * K + j];
    }

    // Load the slice, form the sub-tile sums and exchange the slice totals.
    // Afterwards sh_S (identical bits in every CTA), sh_slice_prefix,
    // sh_all_lastpos and sh_owner are set.
    int xr = 0;  // exchanges done
    auto load_and_exchange = [&]() {
        int lp = -1;
        // all chunks in flight at once, or (RELOAD) batches of 4 chunks (2 when
        // each value is formed from a logit: more registers per chunk)
        constexpr int kBatch = RELOAD ? (LG ? 2 : 4) : kRegChunks;
#pragma unroll
        for (int i0 = 0; i0 < kRegChunks; i0 += kBatch) {
#pragma unroll
            for (int i = i0; i < i0 + kBatch; ++i)
                load_law4x<VEC, LG>(prow, qrow, use_res, v0 + 4 * (int64_t(i) * kAcceptThreads + threadIdx.x), V,
                                    r[i], ps, qs, P.inv_t);
#pragma unroll
            for (int i = i0; i < i0 + kBatch; ++i) {
                const float sm = warp_sum_f((r[i][0] + r[i][1]) + (r[i][2] + r[i][3]));
                if (lane == 0) subsum[i * kAcceptWarps + warp] = sm;
                const int e0 = int(v0) + 4 * (i * kAcceptThreads + int(threadIdx.x));
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (r[i][e] > 0.f) lp = max(lp, e0 + e);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, o));
        if (threadIdx.x == 0) sh_lastpos = -1;
        __syncthreads();
        if (lane == 0 && lp >= 0) atomicMax(&sh_lastpos, lp);
        // slice total: sub-tile st in thread st, a fixed-order pair reduction
        if (threadIdx.x < kRegSub) {
            ff v = ff_make(subsum[threadIdx.x]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v = ff_add(v, ff_shfl_xor(v, o));
            if (lane == 0) wsum[warp] = v;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            ff tot = wsum[0];
#pragma unroll
            for (int w = 1; w < kRegSub / 32; ++w) tot = ff_add(tot, wsum[w]);
            const SliceSummaryFF mine{tot, sh_lastpos};
            for (int c = 0; c < C; ++c) cluster.map_shared_rank(&sh_sums[xr][0], c)[rank] = mine;
        }
        cluster.sync();  // every summary has landed in every CTA; none is read remotely afterwards
        if (threadIdx.x == 0) {
            SliceSummaryFF o[kMaxCluster];
#pragma unroll
            for (int c = 0; c < kMaxCluster; ++c)
                if (c < C) o[c] = sh_sums[xr][c];
            ff S{0.f, 0.f}, prefix{0.f, 0.f};
            int last = -1;
#pragma unroll
            for (int c = 0; c < kMaxCluster; ++c)
                if (c < C) {
                    if (c == rank) prefix = S;
                    S = ff_add(S, o[c].total);
                    last = max(last, o[c].lastpos);
                }
            // the slice holding the first crossing, found identically everywhere
            int owner = -1;
            if (S.hi > 0.f && isfinite(S.hi)) {
                const ff thr = ff_mul_f(S, uK);
                ff run{0.f, 0.f};
#pragma unroll
                for (int c = 0; c < kMaxCluster; ++c)
                    if (c < C && owner < 0) {
                        const ff end = ff_add(run, o[c].total);
                        if (o[c].total.hi > 0.f && ff_gt(end, thr)) owner = c;
                        run = end;
                    }
            }
            sh_S = S;
            sh_slice_prefix = prefix;
            sh_all_lastpos = last;
            sh_owner = owner;
        }
        __syncthreads();
        ++xr;
    };
    load_and_exchange();
    if (!(sh_S.hi > 0.f)) {
        // A positive residual exists whenever rejection is possible; only the
        // rounding of the inputs gets here.  Sample p_j instead.
        if (threadIdx.x == 0) sh_flags |= MXS_DEV_ZERO_RESIDUAL;
        use_res = false;
        qrow = nullptr;
        load_and_exchange();
    }
    const ff S = sh_S;
    const bool no_law = !(S.hi > 0.f) || !isfinite(S.hi);
    const ff thr = ff_mul_f(S, uK);
    const int owner = sh_owner;
    const int writer = (no_law || owner < 0) ? 0 : owner;
    if (rank != writer) return;

    if (no_law) {
        for (int i = threadIdx.x; i <= K; i += blockDim.x) tok[i] = -1;
        if (threadIdx.x == 0) {
            const int f = sh_flags | MXS_DEV_NO_LAW;
            P.n_emitted[b] = 0;
            if (P.row_flags) P.row_flags[b] = f;
            report(P.status, f);
        }
        return;
    }

    // --------------------------- locate the sub-tile where C crosses thr
    if (owner >= 0) {
        // thread st < 128 holds sub-tile st: pair scan over them (every shuffle
        // with its whole warp; the crossing thread only copies its start out)
        ff local{0.f, 0.f}, excl{0.f, 0.f}, start{0.f, 0.f};
        if (threadIdx.x < kRegSub) {
            local = ff_make(subsum[threadIdx.x]);
            const ff inc = warp_scan_ff(local, lane);
            excl = warp_excl_ff(inc, lane);
            if (lane == 31) wsum[warp] = inc;
        }
        __syncthreads();
        if (threadIdx.x < kRegSub) {
            start = sh_slice_prefix;
            for (int w = 0; w < warp; ++w) start = ff_add(start, wsum[w]);
            start = ff_add(start, excl);
            if (local.hi > 0.f && ff_gt(ff_add(start, local), thr)) atomicMin(&sh_tstar, int(threadIdx.x));
        }
        __syncthreads();
        if (threadIdx.x < kRegSub && int(threadIdx.x) == sh_tstar) sh_prefix = start;
        __syncthreads();
    }

    // ------------------- exact position, from the registers that hold it
    const int tstar = sh_tstar;
    const int rescan_warp = (owner >= 0 && tstar != INT_MAX) ? (tstar % kAcceptWarps) : 0;
    if (warp == rescan_warp) {
        int pick = -1;
        ff before{0.f, 0.f}, after{0.f, 0.f};
        bool edge_known = false;
        int flags = sh_flags;
        if (owner >= 0 && tstar != INT_MAX) {
            const int ci = tstar / kAcceptWarps;
            float rr[4] = {0.f, 0.f, 0.f, 0.f};
            if constexpr (RELOAD) {
                // the crossing sub-tile again, from L2 (read moments ago)
                load_law4x<VEC, LG>(prow, qrow, use_res, v0 + 4 * (int64_t(ci) * kAcceptThreads + threadIdx.x), V, rr,
                                    ps, qs, P.inv_t);
            } else {
#pragma unroll
                for (int i = 0; i < kRegChunks; ++i)
                    if (i == ci) {
                        rr[0] = r[i][0]; rr[1] = r[i][1]; rr[2] = r[i][2]; rr[3] = r[i][3];
                    }
            }
            ff c[4];
            c[0] = ff_make(rr[0]);
            c[1] = ff_add(c[0], ff_make(rr[1]));
            c[2] = ff_add(c[1], ff_make(rr[2]));
            c[3] = ff_add(c[2], ff_make(rr[3]));
            const ff lane_inc = warp_scan_ff(c[3], lane);
            const ff base = ff_add(sh_prefix, warp_excl_ff(lane_inc, lane));
            int first = 4;
#pragma unroll
            for (int i = 3; i >= 0; --i)
                if (rr[i] > 0.f && ff_gt(ff_add(base, c[i]), thr)) first = i;
            const int e0 = int(v0) + 4 * (ci * kAcceptThreads + warp * 32);
            const unsigned hit = __ballot_sync(0xffffffffu, first < 4);
            if (hit) {
                const int L = __ffs(int(hit)) - 1;
                const int fi = __shfl_sync(0xffffffffu, first, L);
                ff cv{0.f, 0.f};
                float rv = 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (i == fi) { cv = c[i]; rv = rr[i]; }
                const ff cb = ff_shfl(base, L);
                cv = ff_shfl(cv, L);
                rv = __shfl_sync(0xffffffffu, rv, L);
                pick = e0 + 4 * L + fi;
                after = ff_add(cb, cv);
                before = ff_add(after, ff_make(-rv));
            } else {
                // the sub-tile ends at or below u*S when summed in pairs (a
                // rounding tie with its fp32 sum): its last positive element
                int lp = -1;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (rr[i] > 0.f) lp = 4 * lane + i;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, o));
                pick = e0 + lp;
                flags |= MXS_DEV_NEAR_EDGE;
                edge_known = true;
            }
        } else if (owner >= 0) {
            // the slice ends at or below u*S in this summation order (a rounding
            // tie with its total): its last positive element
            pick = sh_lastpos;
            flags |= MXS_DEV_NEAR_EDGE;
            edge_known = true;
        } else {
            // rounding put u*S at or beyond the last positive mass
            pick = sh_all_lastpos;
            float rl[4];
            const int64_t e = int64_t(pick) & ~int64_t(3);
            load_law4x<false, LG>(prow, qrow, use_res, e, V, rl, ps, qs, P.inv_t);
            after = S;
            before = ff_add(S, ff_make(-rl[pick - e]));
        }
        if (lane == 0) {
            if (!edge_known) {
                // |u - C/S| for the two CDF values around the pick
                const ff d0 = ff_add(before, ff_neg(thr)), d1 = ff_add(after, ff_neg(thr));
                const float e0 = fabsf(d0.hi + d0.lo) / S.hi, e1 = fabsf(d1.hi + d1.lo) / S.hi;
                if (fminf(e0, e1) < float(kNearEdge)) flags |= MXS_DEV_NEAR_EDGE;
            }
            tok[j] = pick;
            P.n_emitted[b] = j + 1;
            if (P.row_flags) P.row_flags[b] = flags;
            report(P.status, flags);
        }
    }
    // emitted drafts, then padding
    for (int i = threadIdx.x; i <= K; i += blockDim.x) {
        if (i < j) tok[i] = P.draft[b * K + i];
        else if (i > j) tok[i] = -1;
    }
}

// Multiprocessor count of the current device, queried once per device.
static cudaError_t sm_count(int& sms) {
    static std::atomic<int> cache[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    sms = cache[dev].load(std::memory_order_relaxed);
    if (sms > 0) return cudaSuccess;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) cache[dev].store(sms, std::memory_order_relaxed);
    return e;
}

// One cluster of C CTAs per row.
static cudaError_t launch_cluster(void (*kern)(AcceptParams), const AcceptParams& P, int64_t B, int C,
                                  size_t smem, cudaStream_t stream) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(unsigned(B * C), 1, 1);
    cfg.blockDim = dim3(kAcceptThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = unsigned(C);
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, P);
}

// The register-resident kernel (V <= 131072), in one of three forms by how
// many CTAs the batch needs (C8 = CTAs per row at 16384 elements each):
//  * B C8 <= SMs / 2: registers kept until the rescan (one CTA per SM);
//  * B C8 <= 2 SMs: reload form, two CTAs per SM, one wave;
//  * beyond: reload form with 32768-element slices (clusters of 4 at
//    V = 128256), so every row is in flight at once.
// Measured at V = 128256: B <= 4 ~0.4 us faster with registers; B = 16
// 19.3 -> 11.9 us (reload); B = 64 47.5 -> 25.3 (reload) -> 19.9 us (wide).
template <bool LG>
static cudaError_t launch_reg(const AcceptParams& P, int64_t B, int64_t V, bool vec, cudaStream_t stream) {
    int C = int((V + kAcceptThreads * 32 - 1) / (kAcceptThreads * 32));
    int sms = 0;
    cudaError_t e = sm_count(sms);
    if (e != cudaSuccess) return e;
    const int64_t ctas = int64_t(B) * C;
    int form = 2 * ctas <= int64_t(sms) ? 0 : (ctas <= 2 * int64_t(sms) ? 1 : 2);
    if (LG && form == 2) form = 1;  // one CTA per SM either way; the wide slice would spill
    if (const char* f = std::getenv("MXS_ACCEPT_FORM")) form = std::atoi(f) == 1 ? 1 : (std::atoi(f) == 2 ? 2 : 0);
    if (int64_t(B) * 4 > int64_t(INT32_MAX)) return cudaErrorInvalidConfiguration;  // grid size
    void (*kern)(AcceptParams);
    if (form == 2) {
        C = int((V + kAcceptThreads * 64 - 1) / (kAcceptThreads * 64));
        kern = vec ? spec_accept_reg_kernel<true, true, 16, LG> : spec_accept_reg_kernel<false, true, 16, LG>;
    } else if (form == 1) {
        kern = vec ? spec_accept_reg_kernel<true, true, 8, LG> : spec_accept_reg_kernel<false, true, 8, LG>;
    } else {
        kern = vec ? spec_accept_reg_kernel<true, false, 8, LG> : spec_accept_reg_kernel<false, false, 8, LG>;
    }
    return launch_cluster(kern, P, B, C, 0, stream);
}

cudaError_t accept_run(const float* p, const float* q, const int32_t* draft, const float* u,
                       int64_t B, int64_t K, int64_t V, int32_t* out_tokens, int32_t* n_emitted,
                       int32_t* row_flags, int32_t* dev_status, cudaStream_t stream) {
    AcceptParams P{};
    P.p = p;
    P.q = q;
    P.draft = draft;
    P.u = u;
    P.V = V;
    P.K = int(K);
    P.nsub = int((V + kSubTile - 1) / kSubTile);
    // cluster size: about 64 sub-tiles (8192 elements) or more per CTA
    int C = (P.nsub + 63) / 64;
    C = C < 1 ? 1 : (C > kMaxCluster ? kMaxCluster : C);
    while (int64_t(B) * C > int64_t(INT32_MAX)) C >>= 1;
    P.per_cta = (P.nsub + C - 1) / C;
    P.out_tokens = out_tokens;
    P.n_emitted = n_emitted;
    P.row_flags = row_flags;
    P.status = dev_status;
    const bool vec = (V % 4 == 0) && (reinterpret_cast<uintptr_t>(p) % 16 == 0) &&
                     (K == 0 || reinterpret_cast<uintptr_t>(q) % 16 == 0);
    if (V <= kRegMaxV && std::getenv("MXS_ACCEPT_STREAMING") == nullptr)
        return launch_reg<false>(P, B, V, vec, stream);
    const size_t smem = size_t(P.per_cta) * sizeof(float);
    void (*kern)(AcceptParams) = vec ? spec_accept_kernel<true> : spec_accept_kernel<false>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (err != cudaSuccess) return err;
    return launch_cluster(kern, P, B, C, smem, stream);
}

cudaError_t accept_logits_run(const float* p_logits, const float* q_logits, const LawStats* pst,
                              const LawStats* qst, float inv_t, const int32_t* draft, const float* u,
                              int64_t B, int64_t K, int64_t V, int32_t* out_tokens, int32_t* n_emitted,
                              int32_t* row_flags, int32_t* dev_status, cudaStream_t stream) {
    AcceptParams P{};
    P.p = p_logits;
    P.q = q_logits;
    P.draft = draft;
    P.u = u;
    P.V = V;
    P.K = int(K);
    P.nsub = int((V + kSubTile - 1) / kSubTile);
    P.out_tokens = out_tokens;
    P.n_emitted = n_emitted;
    P.row_flags = row_flags;
    P.status = dev_status;
    P.pst = pst;
    P.qst = qst;
    P.inv_t = inv_t;
    const bool vec = (V % 4 == 0) && (reinterpret_cast<uintptr_t>(p_logits) % 16 == 0) &&
                     (K == 0 || reinterpret_cast<uintptr_t>(q_logits) % 16 == 0);
    return launch_reg<true>(P, B, V, vec, stream);
}

}  // namespace mxs
