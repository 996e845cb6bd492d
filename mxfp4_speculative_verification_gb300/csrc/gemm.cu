// mxfp4_verify_gemm on sm_103a: Y[M,N] = X[M,K] . dequant(W)^T.
//
// Operation: "Module 11. Speculative Decoding and Quantization", §10 (the
// verification pass is a short, wider decode whose cost is the weight read,
// §1) over MX-FP4 weights (§12; packed [rows, K/2] nibbles + [rows, K/32]
// E8M0 scales with fp32 accumulation as in the MX-FP4 GEMV of "Next-Gen
// Speculative Decoding and FP4 Quantization Shake Up LLM Inference
// Economics").
//
// Design (HBM-bound for M <= 64: every weight byte is read exactly once):
//  * a preparation kernel turns X [M, K] bf16 into fp16 tensor-core
//    fragments (each row scaled by a power of two so that it fits fp16
//    exactly), zeroes the split-K counters and, when needed, realigns the
//    scale rows;
//  * the main kernel is persistent: each CTA streams its work items (a tile
//    of BN weight rows x one K range) through one continuous shared-memory
//    ring, so the pipeline never drains between tiles.  A single GEMM's
//    items go round robin over the CTAs.  A grouped launch orders its GEMMs
//    longest item first and, after a round-robin prefix that fills every
//    ring, its CTAs claim further items one at a time from a counter in
//    global memory: a longest-first list schedule, so that items of
//    different K (a layer's down projection against its other projections)
//    end close together on every SM.  One producer thread issues per 512-k stage two 2-D TMA tensor
//    copies of nibbles (128-byte swizzle, evict-first), one of scales and
//    one bulk copy of the stage's X fragments, all completing on one
//    mbarrier.  Consumer warps each own 16 weight rows: ldmatrix fetches
//    nibbles, the hardware E2M1->fp16 conversion decodes them, and
//    mma.sync m16n8k16 multiplies (weights = MMA rows, candidate positions =
//    MMA columns).  Each 16 x 32 block is accumulated separately and scaled
//    in fp32 by its E8M0 scale, so the block scale is exact for every
//    exponent;
//  * when K is split, each work item writes its partial tile to the
//    workspace and bumps a per-tile counter; the item that completes the
//    count sums all partials in split order (deterministic) and writes Y;
//  * passes of more than 24 rows (and, for a single GEMM, N >= 8192) run
//    instead on the tcgen05 kernel of gemm_umma.cuh, fed by the same
//    preparation kernel in its swizzled tile layout (`use_umma`).
#include <cuda.h>  // CUtensorMap and the tensor-map enums (types only)

#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <vector>

#include <cuda_fp16.h>

#include "mxs_device.cuh"
#include "mxs_internal.h"

namespace mxs {

constexpr int kMaxDevices = 64;
constexpr int kStageBlocks = 16;                 // 16 MX blocks = 512 k per stage
constexpr int kBoxBytes = 128;                   // inner extent of one nibble box (256 k)
constexpr int kFragBytesPerBlockTile = 512;      // one 32-k block x 8 rows of X as fp16 fragments
constexpr int kMaxSplit = 32;
constexpr int64_t kMaxSplitItems = 2048;         // bound on tiles x splits when K is split

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
};

// RG groups of 16 weight rows; KW consumer warps share each group, each
// taking 16/KW of a stage's blocks (KW = 2: one nibble box per warp).
template <int NT, int RG, int KW, int STAGES>
struct GemmCfg {
    static constexpr int BN = 16 * RG;
    static constexpr int NWC = RG * KW;
    static constexpr int kConsumers = 32 * NWC;
    static constexpr int kThreads = kConsumers + 32;
    static constexpr int kBoxW = BN * kBoxBytes;            // one nibble box
    static constexpr int kWBytes = 2 * kBoxW;
    static constexpr int kSBytes = BN * 16;
    static constexpr int kXBytes = kStageBlocks * NT * kFragBytesPerBlockTile;
    static constexpr int kStageBytes = kWBytes + kSBytes + kXBytes;
    static constexpr int kPartPitch = 8 * NT + 1;            // floats per row of the partial tile
    static constexpr int kPartOffset = STAGES * kStageBytes;
    static constexpr int kPartFloats = KW * BN * kPartPitch;  // one partial tile per k-warp
    static constexpr int kBarOffset = kPartOffset + ((kPartFloats * 4 + 15) / 16) * 16;
    static constexpr int kMiscOffset = kBarOffset + 2 * STAGES * 8;
    static constexpr int kItemOffset = kMiscOffset + 16;     // work item of each ring slot
    static constexpr int kSmemBytes = kItemOffset + 16 * ((4 * STAGES + 15) / 16) + 1024;
    // Two CTAs per SM when the shared memory allows them (228 KB per SM, 1 KB
    // reserved per CTA), else 0 (the register budget left to the compiler)
    static constexpr int kMinBlocks = 2 * (kSmemBytes + 1024) <= 233472 ? 2 : 0;
    static_assert(kStageBytes % 1024 == 0, "128-byte swizzled boxes need 1 KB aligned stages");
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                            uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1, const float (&c)[4]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%10, %11, %12, %13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
          "f"(c[3]));
}

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

__device__ __forceinline__ void consumer_bar(int nthreads) {
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// Barrier over the consumer threads that also returns whether v held on any
// of them: the consumers leave their item loop together or not at all.
__device__ __forceinline__ bool consumer_any(int nthreads, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pv, pr;\n\t"
        "setp.ne.u32 pv, %1, 0;\n\t"
        "barrier.cta.red.or.pred pr, 2, %2, pv;\n\t"
        "selp.u32 %0, 1, 0, pr;\n\t}"
        : "=r"(r)
        : "r"(uint32_t(v)), "r"(nthreads)
        : "memory");
    return r != 0;
}

// One consumer warp's share of a stage: 16/KW consecutive blocks (the first
// nbl of them when the stage is short).  w_row: shared address of this
// lane's ldmatrix row in the warp's first nibble box; lm[j]: swizzled
// offset of the lane's 16-byte chunk for block pair j; sgw/sg8w: the scale
// bytes of the warp's blocks for rows g and g+8; xs: the X fragments of the
// warp's first block.
template <int NT, int BOXW, int KW, bool FULL>
__device__ __forceinline__ void consume_stage(float (&acc)[NT][4], uint32_t w_row,
                                              const uint32_t (&lm)[4],
                                              const uint32_t (&sgw)[4 / KW],
                                              const uint32_t (&sg8w)[4 / KW],
                                              const uint4* __restrict__ xs, int lane, int nbl) {
    const float zero[4] = {0.f, 0.f, 0.f, 0.f};
    constexpr int kPairs = kStageBlocks / 2 / KW;  // block pairs per k-warp
#pragma unroll
    for (int bq = 0; bq < kPairs; ++bq) {
        if (!FULL && 2 * bq >= nbl) break;
        uint32_t r0, r1, r2, r3;
        // r0: rows 0-7 blk 2bq, r1: rows 8-15 blk 2bq, r2/r3: blk 2bq+1
        ldmatrix_x4(w_row + (bq >> 2) * BOXW + lm[bq & 3], r0, r1, r2, r3);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int blk = 2 * bq + h;
            if (!FULL && blk >= nbl) break;
            uint32_t ag[4], ag8[4];
            e2m1x8_to_f16x2x4(h ? r2 : r0, ag[0], ag[1], ag[2], ag[3]);
            e2m1x8_to_f16x2x4(h ? r3 : r1, ag8[0], ag8[1], ag8[2], ag8[3]);
            const uint32_t sel = (blk & 3) | ((4 + (blk & 3)) << 4);
            float s_g, s_g8;
            e8m0x2_to_f32x2(__byte_perm(sgw[blk >> 2], sg8w[blk >> 2], sel), s_g, s_g8);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const uint4 xv = xs[(blk * NT + nt) * 32 + lane];
                float d[4];
                mma_16816(d, ag[0], ag8[0], ag[1], ag8[1], xv.x, xv.y, zero);
                mma_16816(d, ag[2], ag8[2], ag[3], ag8[3], xv.z, xv.w, d);
                acc[nt][0] = fmaf(d[0], s_g, acc[nt][0]);
                acc[nt][1] = fmaf(d[1], s_g, acc[nt][1]);
                acc[nt][2] = fmaf(d[2], s_g8, acc[nt][2]);
                acc[nt][3] = fmaf(d[3], s_g8, acc[nt][3]);
            }
        }
    }
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

// Register budget, measured (same GB300, A/B): a single GEMM's short split-K
// items run fastest with the budget set for the CTAs per SM that fit (no
// spills in the per-item path); the grouped launches' long items with the
// compiler's own budget.
template <int NT, int RG, int KW, int STAGES, int G>
__global__ void __launch_bounds__(GemmCfg<NT, RG, KW, STAGES>::kThreads,
                                  G == 1 ? GemmCfg<NT, RG, KW, STAGES>::kMinBlocks : 0)
    mxfp4_gemm_kernel(const __grid_constant__ ProblemSet<G> S) {
    using C = GemmCfg<NT, RG, KW, STAGES>;
    constexpr int NWC = C::NWC;
    extern __shared__ uint8_t smem_raw[];
    // 128-byte-swizzled TMA destinations need 1 KB alignment
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_base & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    const uint32_t smem_base = raw_base + pad;
    const uint32_t full_bar = smem_base + C::kBarOffset;
    const uint32_t empty_bar = full_bar + STAGES * 8;
    float* part = reinterpret_cast<float*>(smem + C::kPartOffset);
    int* sh_last = reinterpret_cast<int*>(smem + C::kMiscOffset);
    // item whose first stage a slot holds (-1: no items left), written by the
    // producer before the slot's full barrier completes
    volatile int* sh_item = reinterpret_cast<volatile int*>(smem + C::kItemOffset);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar + 8 * s, 1);
            mbar_init(empty_bar + 8 * s, NWC);
        }
        mbar_fence_init();
    }
    __syncthreads();
    pdl_trigger();

    if (warp == NWC) {
        // ------------------------------------------------------- producer
        if (lane != 0) return;
        const uint64_t pol_w = policy_evict_first();
        const uint64_t pol_x = policy_evict_last();
        // copies that depend on the preparation kernel are deferred until
        // the first STAGES stages of weights are in flight
        int def_slot[STAGES], def_kb[STAGES], def_nb[STAGES], def_n0[STAGES], def_pi[STAGES];
        int ndef = 0;
        bool waited = false;
        auto issue_dep = [&](int slot, int kb, int nb, int n0, int pi) {
            const Problem& pb = S.p[pi];
            const uint32_t stage = smem_base + slot * C::kStageBytes;
            const uint32_t bar = full_bar + 8 * slot;
            if (pb.sc_from_prep) tma_2d(stage + C::kWBytes, &pb.tm_s, kb, n0, bar, pol_w);
            bulk_g2s(stage + C::kWBytes + C::kSBytes,
                     pb.xf + int64_t(kb) * NT * (kFragBytesPerBlockTile / 2),
                     uint32_t(nb) * NT * kFragBytesPerBlockTile, bar, pol_x);
        };
        int it = 0;
        int last_pi = -1;
        bool ok = true;
        int w = blockIdx.x;
        int taken = 1;  // items this CTA has started
        while (ok && w < S.items) {
            // The next item, one item ahead: the first nstatic of a CTA in
            // round-robin order (enough stages to fill the ring before the
            // preceding kernels finish), then from the counter, which the
            // preceding kernels zero (so only after griddepcontrol.wait).
            int next = -1;
            const bool by_counter = G > 1 && S.sched != nullptr && taken >= S.nstatic;
            auto claim = [&]() {
                next = by_counter ? S.nstatic * int(gridDim.x) + atomicAdd(S.sched, 1) : w + int(gridDim.x);
            };
            const int pi = find_problem(S, w);
            const Problem& pb = S.p[pi];
            if (pi != last_pi) {
                prefetch_tmap(&pb.tm_w);
                prefetch_tmap(&pb.tm_s);
                last_pi = pi;
            }
            const ItemRange R = item_range(pb, w - pb.item_begin);
            const int n0 = R.tile * C::BN;
            for (int i = 0; i < R.nst; ++i, ++it) {
                const int slot = it % STAGES;
                if (it >= STAGES &&
                    !mbar_wait(empty_bar + 8 * slot, ((it / STAGES) - 1) & 1, S.status)) {
                    ok = false;
                    break;
                }
                const int kb = R.kb0 + i * kStageBlocks;
                const int nb = min(kStageBlocks, R.kb1 - kb);
                const uint32_t stage = smem_base + slot * C::kStageBytes;
                const uint32_t bar = full_bar + 8 * slot;
                if (G > 1 && i == 0) sh_item[slot] = w;
                mbar_arrive_expect_tx(bar, uint32_t(C::kWBytes + C::kSBytes) +
                                               uint32_t(nb) * NT * kFragBytesPerBlockTile);
                tma_2d(stage, &pb.tm_w, kb * 16, n0, bar, pol_w);
                tma_2d(stage + C::kBoxW, &pb.tm_w, kb * 16 + kBoxBytes, n0, bar, pol_w);
                if (!pb.sc_from_prep) tma_2d(stage + C::kWBytes, &pb.tm_s, kb, n0, bar, pol_w);
                if (waited) {
                    issue_dep(slot, kb, nb, n0, pi);
                } else {
                    def_slot[ndef] = slot;
                    def_kb[ndef] = kb;
                    def_nb[ndef] = nb;
                    def_n0[ndef] = n0;
                    def_pi[ndef] = pi;
                    ++ndef;
                    if (ndef == STAGES) {
                        pdl_wait();
                        waited = true;
                        for (int d = 0; d < ndef; ++d)
                            issue_dep(def_slot[d], def_kb[d], def_nb[d], def_n0[d], def_pi[d]);
                    }
                }
                if (next < 0 && (waited || !by_counter)) claim();
            }
            if (!ok) break;
            if (next < 0) {
                if (!waited) {
                    pdl_wait();
                    waited = true;
                    for (int d = 0; d < ndef; ++d)
                        issue_dep(def_slot[d], def_kb[d], def_nb[d], def_n0[d], def_pi[d]);
                }
                claim();
            }
            w = next;
            ++taken;
        }
        if (!waited) {
            pdl_wait();
            for (int d = 0; d < ndef; ++d)
                issue_dep(def_slot[d], def_kb[d], def_nb[d], def_n0[d], def_pi[d]);
        }
        // never leave a copy in flight: wait (bounded) for the last phase of
        // every slot filled
        for (int j = max(0, it - STAGES); j < it; ++j)
            mbar_wait(full_bar + 8 * (j % STAGES), (j / STAGES) & 1, S.status);
        // end of the item stream (after the waits above, which read the
        // slots' current phases): a slot whose barrier completes without copies
        if (G > 1 && ok) {
            const int slot = it % STAGES;
            if (it < STAGES || mbar_wait(empty_bar + 8 * slot, ((it / STAGES) - 1) & 1, S.status)) {
                sh_item[slot] = -1;
                mbar_arrive(full_bar + 8 * slot);
            }
        }
        return;
    }

    // ----------------------------------------------------------- consumers
    const int g = lane >> 2, t = lane & 3;
    const int rbase = (warp % RG) * 16;
    const int kw = warp / RG;
    const int mi = lane >> 3, ri = lane & 7;
    const int lrow = rbase + ri + 8 * (mi & 1);
    uint32_t lm[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) lm[j] = uint32_t(((2 * j + (mi >> 1)) ^ ri) << 4);
    const int M = S.M;
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    bool waited = false;
    int it = 0;
    bool ok = true;
    // a single GEMM: the static round robin; grouped: the item each first
    // stage's slot names
    for (int ws = blockIdx.x;; ws += gridDim.x) {
        int w = ws;
        if constexpr (G == 1) {
            if (w >= S.items) break;
        } else {
            w = -1;
            if (ok) {
                const int slot = it % STAGES;
                if (mbar_wait(full_bar + 8 * slot, (it / STAGES) & 1, S.status)) w = sh_item[slot];
                else ok = false;
            }
            __syncwarp();
            if (consumer_any(C::kConsumers, w < 0)) break;
        }
        const Problem& P = S.p[find_problem(S, w)];
        const int wl = w - P.item_begin;  // item index within its GEMM
        const ItemRange R = item_range(P, wl);
        const int64_t n0 = int64_t(R.tile) * C::BN;
        const int rows = int(P.N - n0 < int64_t(C::BN) ? P.N - n0 : int64_t(C::BN));
        for (int i = 0; ok && i < R.nst; ++i, ++it) {
            const int slot = it % STAGES;
            if (!mbar_wait(full_bar + 8 * slot, (it / STAGES) & 1, S.status)) {
                ok = false;
                break;
            }
            const int nb = min(kStageBlocks, R.kb1 - (R.kb0 + i * kStageBlocks));
            const uint8_t* stage = smem + slot * C::kStageBytes;
            constexpr int kWords = 4 / KW;  // scale words (4 blocks each) per k-warp
            const uint32_t* s_row = reinterpret_cast<const uint32_t*>(stage + C::kWBytes);
            uint32_t sgw[kWords], sg8w[kWords];
#pragma unroll
            for (int q = 0; q < kWords; ++q) {
                sgw[q] = s_row[(rbase + g) * 4 + kw * kWords + q];
                sg8w[q] = s_row[(rbase + g + 8) * 4 + kw * kWords + q];
            }
            constexpr int kBlocksPerWarp = kStageBlocks / KW;
            const uint4* xs = reinterpret_cast<const uint4*>(stage + C::kWBytes + C::kSBytes) +
                              kw * kBlocksPerWarp * NT * 32;
            // k-warp kw starts at block kw*16/KW: box (kw*16/KW)/8, chunk pairs from 0
            const uint32_t w_row = smem_base + slot * C::kStageBytes + uint32_t(lrow) * kBoxBytes +
                                   uint32_t((kw * kBlocksPerWarp) / 8) * C::kBoxW;
            const int nbl = nb - kw * kBlocksPerWarp;
            if (nb == kStageBlocks)
                consume_stage<NT, C::kBoxW, KW, true>(acc, w_row, lm, sgw, sg8w, xs, lane, nbl);
            else
                consume_stage<NT, C::kBoxW, KW, false>(acc, w_row, lm, sgw, sg8w, xs, lane, nbl);
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar + 8 * slot);
        }

        // --------------------------------------------- epilogue of one item
        consumer_bar(C::kConsumers);  // the previous item's partial tile is consumed
        {
            const int r = rbase + g;
            float* pk = part + kw * (C::BN * C::kPartPitch);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                pk[r * C::kPartPitch + nt * 8 + 2 * t] = acc[nt][0];
                pk[r * C::kPartPitch + nt * 8 + 2 * t + 1] = acc[nt][1];
                pk[(r + 8) * C::kPartPitch + nt * 8 + 2 * t] = acc[nt][2];
                pk[(r + 8) * C::kPartPitch + nt * 8 + 2 * t + 1] = acc[nt][3];
                acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
            }
        }
        consumer_bar(C::kConsumers);
        // the item's sum over its k-warps, in a fixed order
        auto tile_val = [&](int r, int m) {
            float v = part[r * C::kPartPitch + m];
#pragma unroll
            for (int q = 1; q < KW; ++q) v += part[q * (C::BN * C::kPartPitch) + r * C::kPartPitch + m];
            return v;
        };
        if (!waited) {
            pdl_wait();  // Y, the counters and xun belong to the preceding kernels until now
            waited = true;
        }
        if (P.nsplit == 1) {
            for (int o = threadIdx.x; o < C::BN * M; o += C::kConsumers) {
                const int r = o % C::BN, m = o / C::BN;
                if (r < rows) P.y[int64_t(m) * P.N + n0 + r] = tile_val(r, m) * P.xun[m];
            }
        } else {
            float* mine = P.part + int64_t(wl) * M * C::BN;
            for (int o = threadIdx.x; o < C::BN * M; o += C::kConsumers) {
                const int r = o % C::BN, m = o / C::BN;
                __stcg(mine + int64_t(m) * C::BN + r, tile_val(r, m));
            }
            __threadfence();
            consumer_bar(C::kConsumers);
            if (threadIdx.x == 0) *sh_last = (atomicAdd(P.counters + R.tile, 1) == P.nsplit - 1);
            consumer_bar(C::kConsumers);
            if (*sh_last) {
                __threadfence();
                for (int o = threadIdx.x; o < C::BN * M; o += C::kConsumers) {
                    const int r = o % C::BN, m = o / C::BN;
                    if (r < rows) {
                        float s = 0.f;
                        for (int q = 0; q < P.nsplit; ++q)
                            s += __ldcg(P.part + (int64_t(q) * P.ntiles + R.tile) * M * C::BN +
                                        int64_t(m) * C::BN + r);
                        P.y[int64_t(m) * P.N + n0 + r] = s * P.xun[m];
                    }
                }
                if (threadIdx.x == 0) P.counters[R.tile] = 0;  // ready for the next call
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Preparation: X bf16 [M, K] -> fp16 fragments and per-row unscale factors;
// zeroed split-K counters; optional copy of the scale rows into 16-byte
// aligned rows.
//
// Row m is multiplied by 2^sh with sh = 142 - (biased exponent of max|x|),
// which puts max|x| in [2^15, 2^16): fp16 then holds every element within
// 2^29 of the maximum exactly.  The GEMM multiplies its output by 2^-sh.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float pow2f_exact(int e) {
    // 2^e as fp32 for e in [-149, 127]
    if (e >= -126) return __uint_as_float(uint32_t(e + 127) << 23);
    return __uint_as_float(1u << (e + 149));
}

#include "gemm_umma.cuh"

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

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

static int tiles_nt(int mc) {  // fragment tiles of 8 rows used for a pass of mc rows
    const int nt = (mc + 7) / 8;
    return nt > 4 ? 8 : nt;
}
static int bn_for_nt(int nt) { return (nt == 3 || nt == 4) ? 128 : 64; }

// Largest split-K work-item count the launcher may pick (0 if it never splits).
static int64_t split_items_cap(int64_t N, int64_t K, int bn) {
    const int64_t ntiles = (N + bn - 1) / bn;
    const int64_t stages = (K / 32 + kStageBlocks - 1) / kStageBlocks;
    const int64_t ns = std::min<int64_t>(
        {int64_t(kMaxSplit), stages, std::max<int64_t>(1, kMaxSplitItems / ntiles)});
    return ns > 1 ? ntiles * ns : 0;
}

GemmWorkspace gemm_workspace_layout(int64_t M, int64_t N, int64_t K, bool scales_aligned) {
    GemmWorkspace w{};
    const int64_t nblk = K / 32;
    const int64_t mc = std::min<int64_t>(M, kGemmMaxRowsPerPass);
    w.repack_scales = !(K % 512 == 0 && scales_aligned);
    w.sc_pitch = w.repack_scales ? int(align_up(size_t(nblk), 16)) : int(nblk);
    size_t off = 0;
    w.xf_off = off;
    off = align_up(off + size_t(kGemmMaxRowsPerPass) * align_up(size_t(K), 512) * 2, 256);
    w.xun_off = off;
    off = align_up(off + kGemmMaxRowsPerPass * sizeof(float), 256);
    // counters and partial tiles, sized for either tile height a pass may use
    int64_t ncnt = 0, part = 0;
    for (int bn : {64, 128}) {
        const int64_t cap = split_items_cap(N, K, bn);
        if (cap > 0) {
            ncnt = std::max<int64_t>(ncnt, (N + bn - 1) / bn);
            part = std::max<int64_t>(part, cap * mc * bn);
        }
    }
    w.cnt_off = off;
    w.n_counters = int(ncnt);
    off = align_up(off + size_t(ncnt) * sizeof(int), 256);
    w.part_off = off;
    off = align_up(off + size_t(part) * sizeof(float), 256);
    w.sc_off = off;
    if (w.repack_scales) off = align_up(off + size_t(N) * size_t(w.sc_pitch), 256);
    w.bytes = off;
    return w;
}

static int env_int(const char* name, int dflt) {
    const char* v = std::getenv(name);
    return v ? std::atoi(v) : dflt;
}

// cuTensorMapEncodeTiled, fetched from the driver through the runtime.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static std::atomic<EncodeTiledFn> fn{nullptr};
    EncodeTiledFn f = fn.load(std::memory_order_acquire);
    if (!f) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        f = reinterpret_cast<EncodeTiledFn>(p);
        fn.store(f, std::memory_order_release);
    }
    return f;
}

// 2-D uint8 tensor map over a [rows, cols] byte matrix with the given row pitch.
static bool make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols,
                     int64_t pitch, uint32_t box_cols, uint32_t box_rows, bool swizzle128) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(pitch)};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    std::memset(map, 0, sizeof(*map));
    return f(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Per-device launch facts of one kernel instantiation, computed on first use.
struct LaunchFacts {
    std::atomic<int> sms[kMaxDevices];
    std::atomic<int> occ[kMaxDevices];
};

// Split of K: the count whose busiest CTA streams the fewest stages, with a
// small charge per extra work item for its partial-tile round trip.
static void choose_split(int64_t ntiles, int stages_total, int64_t grid_cap, int64_t items_cap,
                         int& nsplit, int& per_split) {
    double best = 1e300;
    nsplit = 1;
    per_split = stages_total;
    const int max_ns = int(std::min<int64_t>(kMaxSplit, stages_total));
    for (int ns = 1; ns <= max_ns; ++ns) {
        const int sps = (stages_total + ns - 1) / ns;
        const int nse = (stages_total + sps - 1) / sps;  // splits actually used
        if (nse != ns) continue;
        const int64_t items = ntiles * ns;
        if (ns > 1 && items > items_cap) break;
        const int64_t grid = std::min<int64_t>(items, grid_cap);
        const double per_cta = double((items + grid - 1) / grid);
        const double cost = per_cta * (sps + (ns > 1 ? 0.35 : 0.0));
        if (cost < best - 1e-9) {
            best = cost;
            nsplit = ns;
            per_split = sps;
        }
    }
}

// One GEMM as the host describes it before the launch is planned.
struct HostGemm {
    const uint8_t* nib;
    const uint8_t* sc;   // the scale rows actually streamed (in place or realigned)
    int sc_pitch;
    bool sc_from_prep;
    const uint16_t* xf;
    const float* xun;
    float* y;
    float* part;
    int* counters;
    int64_t N, K;
    int64_t items_cap;   // 0: never split K
};

// Fill the launch's problem table for tiles of BN rows.
template <int G>
static cudaError_t build_problems(ProblemSet<G>& S, const HostGemm* gs, int count, int M,
                                  int32_t* status, int BN, int64_t resident, int* sched) {
    std::memset(&S, 0, sizeof(S));
    S.count = count;
    S.M = M;
    S.status = status;
    S.sched = sched;
    int64_t items = 0;
    const int forced = env_int("MXS_GEMM_SPLITS", 0);
    for (int i = 0; i < count; ++i) {
        const HostGemm& h = gs[i];
        Problem& p = S.p[i];
        p.xf = h.xf;
        p.xun = h.xun;
        p.y = h.y;
        p.part = h.part;
        p.counters = h.counters;
        p.N = h.N;
        p.nblk = int(h.K / 32);
        p.ntiles = int((h.N + BN - 1) / BN);
        p.sc_from_prep = h.sc_from_prep ? 1 : 0;
        p.sc = h.sc;
        p.sc_pitch = h.sc_pitch;
        const int stages_total = (p.nblk + kStageBlocks - 1) / kStageBlocks;
        p.nsplit = 1;
        p.stages_per_split = stages_total;
        if (h.items_cap > 0) {
            choose_split(p.ntiles, stages_total, resident, h.items_cap, p.nsplit, p.stages_per_split);
            if (forced > 0) {
                int ns = std::min(forced, stages_total);
                const int sps = (stages_total + ns - 1) / ns;
                ns = (stages_total + sps - 1) / sps;
                if (ns == 1 || int64_t(p.ntiles) * ns <= h.items_cap) {
                    p.nsplit = ns;
                    p.stages_per_split = sps;
                }
            }
        }
        p.item_begin = int(items);
        items += int64_t(p.ntiles) * p.nsplit;
        if (items > INT32_MAX) return cudaErrorInvalidValue;
        if (!make_map(&p.tm_w, h.nib, h.N, h.K / 2, h.K / 2, kBoxBytes, uint32_t(BN), true))
            return cudaErrorInvalidValue;
        if (!make_map(&p.tm_s, h.sc, h.N, p.nblk, h.sc_pitch, 16, uint32_t(BN), false))
            return cudaErrorInvalidValue;
    }
    S.items = int(items);
    return cudaSuccess;
}

// SM count and resident CTAs per SM of one kernel, cached per device.
template <typename Kern>
static cudaError_t launch_facts(LaunchFacts& facts, Kern kern, int threads, int smem, int& sms,
                                int& occ) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    sms = facts.sms[dev].load(std::memory_order_acquire);
    occ = facts.occ[dev].load(std::memory_order_acquire);
    if (sms > 0 && occ > 0) return cudaSuccess;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, smem);
    if (err != cudaSuccess) return err;
    if (occ < 1) occ = 1;
    facts.occ[dev].store(occ, std::memory_order_release);
    facts.sms[dev].store(sms, std::memory_order_release);
    return cudaSuccess;
}

// Persistent launch with programmatic dependent launch enabled.
template <typename Kern, typename Set>
static cudaError_t launch_persistent(Kern kern, const Set& S, int threads, int smem, int64_t grid,
                                     cudaStream_t stream) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(unsigned(grid), 1, 1);
    cfg.blockDim = dim3(unsigned(threads), 1, 1);
    cfg.dynamicSmemBytes = size_t(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, S);
}

template <int NT, int RG, int KW, int STAGES, int G>
static cudaError_t launch_main(const HostGemm* gs, int count, int M, int32_t* status,
                               int* sched, cudaStream_t stream) {
    using C = GemmCfg<NT, RG, KW, STAGES>;
    auto kern = mxfp4_gemm_kernel<NT, RG, KW, STAGES, G>;
    static LaunchFacts facts;
    int sms = 0, occ = 0;
    cudaError_t err = launch_facts(facts, kern, C::kThreads, C::kSmemBytes, sms, occ);
    if (err != cudaSuccess) return err;
    const int64_t resident = int64_t(sms) * occ;
    // the problem table lives in the (large) kernel parameter block
    static thread_local ProblemSet<G>* S_buf = nullptr;
    if (!S_buf) S_buf = new ProblemSet<G>;
    err = build_problems(*S_buf, gs, count, M, status, C::BN, resident, sched);
    if (err != cudaSuccess) return err;
    // round-robin items per CTA before claiming: enough for STAGES stages
    int min_nst = STAGES;
    for (int i = 0; i < count; ++i) {
        const Problem& p = S_buf->p[i];
        const int total = (p.nblk + kStageBlocks - 1) / kStageBlocks;
        const int last = total - (p.nsplit - 1) * p.stages_per_split;
        min_nst = std::min(min_nst, std::min(p.stages_per_split, last));
    }
    S_buf->nstatic = (STAGES + min_nst - 1) / min_nst;
    const int64_t grid = std::min<int64_t>(S_buf->items, resident);
    return launch_persistent(kern, *S_buf, C::kThreads, C::kSmemBytes, grid, stream);
}

// Kernel shape for a pass of M <= 64 rows: NT fragment tiles of 8 rows.
template <int G>
static cudaError_t launch_main_nt(int NT, const HostGemm* gs, int count, int M, int32_t* status,
                                  int* sched, cudaStream_t stream) {
    switch (NT) {
        case 1: return launch_main<1, 4, 2, 4, G>(gs, count, M, status, sched, stream);
        case 2: return launch_main<2, 4, 2, 3, G>(gs, count, M, status, sched, stream);
        case 3: return launch_main<3, 8, 2, 3, G>(gs, count, M, status, sched, stream);
        case 4: return launch_main<4, 8, 2, 2, G>(gs, count, M, status, sched, stream);
        default: return launch_main<8, 4, 2, 2, G>(gs, count, M, status, sched, stream);
    }
}

// tcgen05 kernel: one CTA per SM, whole 128-row tiles (K is never split).
template <int NPAD, int STAGES, int G>
static cudaError_t launch_umma(const HostGemm* gs, int count, int M, int32_t* status,
                               cudaStream_t stream) {
    using C = UCfg<NPAD, STAGES>;
    auto kern = mxfp4_gemm_umma_kernel<NPAD, STAGES, G>;
    static LaunchFacts facts;
    int sms = 0, occ = 0;
    cudaError_t err = launch_facts(facts, kern, kUThreads, C::kSmemBytes, sms, occ);
    if (err != cudaSuccess) return err;
    static thread_local ProblemSet<G>* S_buf = nullptr;
    if (!S_buf) S_buf = new ProblemSet<G>;
    HostGemm tmp[G];
    for (int i = 0; i < count; ++i) {
        tmp[i] = gs[i];
        tmp[i].items_cap = 0;
    }
    err = build_problems(*S_buf, tmp, count, M, status, kUBN, int64_t(sms), nullptr);
    if (err != cudaSuccess) return err;
    const int64_t grid = std::min<int64_t>(S_buf->items, int64_t(sms));
    return launch_persistent(kern, *S_buf, kUThreads, C::kSmemBytes, grid, stream);
}

// Rows of the X tile fed to the tensor cores for a pass of mc rows (MMA N).
static int umma_npad(int mc) { return std::max(16, (mc + 15) / 16 * 16); }

template <int G>
static cudaError_t launch_umma_np(int npad, const HostGemm* gs, int count, int M, int32_t* status,
                                  cudaStream_t stream) {
    switch (npad) {
        case 16: return launch_umma<16, 4, G>(gs, count, M, status, stream);
        case 32: return launch_umma<32, 3, G>(gs, count, M, status, stream);
        case 48: return launch_umma<48, 2, G>(gs, count, M, status, stream);
        default: return launch_umma<64, 2, G>(gs, count, M, status, stream);
    }
}

// Which kernel a pass of mc rows uses.  mma.sync (legacy tensor path) is
// faster up to 24 rows; beyond that its m16n8k16 issue rate, not HBM,
// bounds it and the tcgen05 kernel takes over.  MXS_GEMM_PATH=mma|umma
// forces one (umma needs more than 8 rows).
static bool use_umma(int mc, int64_t tiles128, bool grouped) {
    const char* path = std::getenv("MXS_GEMM_PATH");
    if (path && std::strcmp(path, "mma") == 0) return false;
    if (path && std::strcmp(path, "umma") == 0) return mc > 8;
    // the tcgen05 kernel never splits K: a lone GEMM needs enough 128-row tiles
    return mc > 24 && (grouped || tiles128 >= 64);
}

// The claim counter a grouped launch of the mma.sync kernel uses, or null for
// the static round-robin order (MXS_GEMM_SCHED=static, for comparison).  A
// single GEMM always takes the static order: its items are uniform, and its
// split-K items (one or two stages) would expose the claim's latency.
static int* sched_or_null(int* counter) {
    const char* v = std::getenv("MXS_GEMM_SCHED");
    return (v && std::strcmp(v, "static") == 0) ? nullptr : counter;
}

static cudaError_t launch_prep(const PrepSet& Q, cudaStream_t stream) {
    cudaLaunchConfig_t cfg{};
    const int rows = Q.umma_npad > 0 ? Q.umma_npad : 8 * Q.NT;
    cfg.gridDim = dim3(unsigned(Q.njobs * rows + 1 + Q.repack_ctas), 1, 1);
    cfg.blockDim = dim3(kPrepThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, mxfp4_gemm_prep_kernel, Q);
}

cudaError_t gemm_run(const uint16_t* x, const uint8_t* nibbles, const uint8_t* scales, float* y,
                     int64_t M, int64_t N, int64_t K, void* workspace, const GemmWorkspace& ws,
                     int32_t* dev_status, cudaStream_t stream) {
    uint8_t* wsb = static_cast<uint8_t*>(workspace);
    uint16_t* xf = reinterpret_cast<uint16_t*>(wsb + ws.xf_off);
    float* xun = reinterpret_cast<float*>(wsb + ws.xun_off);
    int* counters = reinterpret_cast<int*>(wsb + ws.cnt_off);
    float* part = reinterpret_cast<float*>(wsb + ws.part_off);
    uint8_t* sc_aligned = ws.repack_scales ? wsb + ws.sc_off : nullptr;
    const int nblk = int(K / 32);
    const int64_t mc0 = std::min<int64_t>(M, kGemmMaxRowsPerPass);
    for (int64_t m0 = 0; m0 < M; m0 += kGemmMaxRowsPerPass) {
        const int mc = int(std::min<int64_t>(kGemmMaxRowsPerPass, M - m0));
        const int NT = tiles_nt(mc);
        const int bn = bn_for_nt(NT);
        // the workspace holds partial tiles for mc0 rows and tile height bn
        int64_t items_cap = split_items_cap(N, K, bn);
        if (ws.n_counters < (N + bn - 1) / bn || mc > mc0) items_cap = 0;
        const bool umma = use_umma(mc, (N + kUBN - 1) / kUBN, false);
        // the scales are realigned once, by the first pass
        const bool repack = ws.repack_scales && m0 == 0;
        PrepSet Q{};
        Q.job[0].x = x + m0 * K;
        Q.job[0].xf = xf;
        Q.job[0].xun = xun;
        Q.job[0].K = int(K);
        Q.njobs = 1;
        Q.M = mc;
        Q.NT = NT;
        Q.umma_npad = umma ? umma_npad(mc) : 0;
        Q.counters = counters;
        Q.ncounters = ws.n_counters;
        if (repack) {
            Q.sc_in = scales;
            Q.N = N;
            Q.nblk = nblk;
            Q.sc_pitch = ws.sc_pitch;
            Q.sc_out = sc_aligned;
            Q.repack_ctas = int(std::min<int64_t>((N * ws.sc_pitch + kPrepThreads - 1) / kPrepThreads, 1024));
        }
        cudaError_t err = launch_prep(Q, stream);
        if (err != cudaSuccess) return err;
        HostGemm h{};
        h.nib = nibbles;
        h.sc = ws.repack_scales ? sc_aligned : scales;
        h.sc_pitch = ws.sc_pitch;
        h.sc_from_prep = repack;
        h.xf = xf;
        h.xun = xun;
        h.y = y + m0 * N;
        h.part = part;
        h.counters = counters;
        h.N = N;
        h.K = K;
        h.items_cap = items_cap;
        err = umma ? launch_umma_np<1>(umma_npad(mc), &h, 1, mc, dev_status, stream)
                   : launch_main_nt<1>(NT, &h, 1, mc, dev_status, nullptr, stream);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

// ------------------------------------------------------------------ grouped
// Independent GEMMs sharing M <= 64: each distinct X is converted once, then
// persistent launches of up to kGroupMax GEMMs stream every weight matrix
// through the same shared-memory ring.
constexpr int kGroupMax = 64;

// Bytes of one prepared X (either layout) for passes of at most mc0 rows.
static size_t xf_bytes(int mc0, int64_t K) {
    const int rows = std::max(8 * tiles_nt(mc0), umma_npad(mc0));
    return size_t(rows) * align_up(size_t(K), 512) * 2;
}

size_t gemm_grouped_workspace(const GroupedGemm* gs, int count, int64_t M) {
    const int mc0 = int(std::min<int64_t>(M, kGemmMaxRowsPerPass));
    size_t off = 0;
    for (int i = 0; i < count; ++i) {
        bool seen = false;
        for (int j = 0; j < i && !seen; ++j) seen = gs[j].x == gs[i].x && gs[j].K == gs[i].K;
        if (seen) continue;
        off = align_up(off + xf_bytes(mc0, gs[i].K), 256);
        off = align_up(off + kGemmMaxRowsPerPass * sizeof(float), 256);
    }
    // one item claim counter per launch of a pass
    return align_up(off + size_t((count + kGroupMax - 1) / kGroupMax) * sizeof(int), 256);
}

cudaError_t gemm_grouped_run(const GroupedGemm* gs, int count, int64_t M, void* workspace,
                             int32_t* dev_status, cudaStream_t stream) {
    uint8_t* wsb = static_cast<uint8_t*>(workspace);
    const int mc0 = int(std::min<int64_t>(M, kGemmMaxRowsPerPass));
    // distinct activations, in first-use order; X space sized for passes of mc0 rows
    std::vector<int> xid(count);
    std::vector<PrepJob> jobs;
    size_t off = 0;
    for (int i = 0; i < count; ++i) {
        int found = -1;
        for (int j = 0; j < int(jobs.size()); ++j)
            if (jobs[j].x == gs[i].x && jobs[j].K == int(gs[i].K)) found = j;
        if (found < 0) {
            PrepJob J{};
            J.x = gs[i].x;
            J.K = int(gs[i].K);
            J.xf = reinterpret_cast<uint16_t*>(wsb + off);
            off = align_up(off + xf_bytes(mc0, gs[i].K), 256);
            J.xun = reinterpret_cast<float*>(wsb + off);
            off = align_up(off + kGemmMaxRowsPerPass * sizeof(float), 256);
            found = int(jobs.size());
            jobs.push_back(J);
        }
        xid[i] = found;
    }
    int* sched = reinterpret_cast<int*>(wsb + off);  // one claim counter per launch of a pass
    const int nlaunch = (count + kGroupMax - 1) / kGroupMax;
    std::vector<HostGemm> hs(count);
    // rows are processed 64 at a time; each pass converts its rows of every
    // distinct X, then streams every weight matrix once
    for (int64_t m0 = 0; m0 < M; m0 += kGemmMaxRowsPerPass) {
        const int mc = int(std::min<int64_t>(kGemmMaxRowsPerPass, M - m0));
        const int NT = tiles_nt(mc);
        const bool umma = use_umma(mc, 0, true);
        for (size_t j0 = 0; j0 < jobs.size(); j0 += kPrepMaxJobs) {
            PrepSet Q{};
            Q.njobs = int(std::min<size_t>(kPrepMaxJobs, jobs.size() - j0));
            for (int q = 0; q < Q.njobs; ++q) {
                Q.job[q] = jobs[j0 + q];
                Q.job[q].x = jobs[j0 + q].x + m0 * jobs[j0 + q].K;
            }
            Q.M = mc;
            Q.NT = NT;
            Q.umma_npad = umma ? umma_npad(mc) : 0;
            if (j0 == 0) {
                Q.counters = sched;
                Q.ncounters = nlaunch;
            }
            cudaError_t err = launch_prep(Q, stream);
            if (err != cudaSuccess) return err;
        }
        for (int i = 0; i < count; ++i) {
            HostGemm& h = hs[i];
            h = HostGemm{};
            h.nib = gs[i].nibbles;
            h.sc = gs[i].scales;
            h.sc_pitch = int(gs[i].K / 32);
            h.sc_from_prep = false;
            h.xf = jobs[xid[i]].xf;
            h.xun = jobs[xid[i]].xun;
            h.y = gs[i].y + m0 * gs[i].N;
            h.N = gs[i].N;
            h.K = gs[i].K;
            h.items_cap = 0;
        }
        // balanced launches of at most kGroupMax GEMMs
        for (int l = 0; l < nlaunch; ++l) {
            const int b = int(int64_t(count) * l / nlaunch);
            const int e = int(int64_t(count) * (l + 1) / nlaunch);
            int* claim = umma ? nullptr : sched_or_null(sched + l);
            // claimed in table order: longest items (largest K) first
            if (claim)
                std::stable_sort(hs.begin() + b, hs.begin() + e,
                                 [](const HostGemm& u, const HostGemm& v) { return u.K > v.K; });
            cudaError_t err =
                umma ? launch_umma_np<kGroupMax>(umma_npad(mc), hs.data() + b, e - b, mc, dev_status, stream)
                     : launch_main_nt<kGroupMax>(NT, hs.data() + b, e - b, mc, dev_status, claim, stream);
            if (err != cudaSuccess) return err;
        }
    }
    return cudaSuccess;
}

}  // namespace mxs
