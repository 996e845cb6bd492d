// The mma.sync verify-GEMM kernel (passes of at most 8 rows by default; the design is
// described at the top of gemm.cu), included by gemm.cu inside namespace mxs.

// RG groups of 16 weight rows; KW consumer warps share each group, each
// taking 16/KW of a stage's blocks (KW = 2: one nibble box per warp).
// NV: NVFP4 weights (one E4M3 scale per 16 k, 32 scale bytes per row per
// 512-k stage) instead of MXFP4 (one E8M0 scale per 32 k, 16 bytes).
template <int NT, int RG, int KW, int STAGES, bool NV = false>
struct GemmCfg {
    static constexpr int BN = 16 * RG;
    static constexpr int NWC = RG * KW;
    static constexpr int kConsumers = 32 * NWC;
    static constexpr int kThreads = kConsumers + 32;
    static constexpr int kBoxW = BN * kBoxBytes;            // one nibble box
    static constexpr int kWBytes = 2 * kBoxW;
    static constexpr int kSBytes = BN * (NV ? 32 : 16);
    static constexpr int kScaleWords = NV ? 8 : 4;          // 32-bit scale words per row per stage
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

__device__ __forceinline__ uint32_t hmul2_f16(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// An E4M3 byte as an f16x2 pair {s, s} (exact: every E4M3 value is an fp16 value).
__device__ __forceinline__ uint32_t e4m3_to_f16x2_pair(uint32_t byte) {
    uint32_t out;
    const uint32_t two = byte | (byte << 8);
    asm("{\n .reg .b16 t;\n cvt.u16.u32 t, %1;\n cvt.rn.f16x2.e4m3x2 %0, t;\n}\n" : "=r"(out) : "r"(two));
    return out;
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
//
// NV: each lane's 8 decoded codes of a 32-k block lie in one 16-element NVFP4
// block (codes 8t .. 8t + 7 for t = lane % 4), so they are multiplied by that
// block's E4M3 scale in fp16 before the MMA (E2M1 x E4M3 has at most 6
// significant bits and lies in [2^-10, 2688]: exact), and the MMAs accumulate
// straight into acc.
template <int NT, int BOXW, int KW, bool FULL, bool NV = false>
__device__ __forceinline__ void consume_stage(float (&acc)[NT][4], uint32_t w_row,
                                              const uint32_t (&lm)[4],
                                              const uint32_t (&sgw)[(NV ? 8 : 4) / KW],
                                              const uint32_t (&sg8w)[(NV ? 8 : 4) / KW],
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
            if constexpr (NV) {
                const int bi = 2 * blk + ((lane & 3) >> 1);  // this lane's NVFP4 block in the warp's share
                const uint32_t sh = 8u * uint32_t(bi & 3);
                const uint32_t s2 = e4m3_to_f16x2_pair((sgw[bi >> 2] >> sh) & 0xFFu);
                const uint32_t s28 = e4m3_to_f16x2_pair((sg8w[bi >> 2] >> sh) & 0xFFu);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    ag[i] = hmul2_f16(ag[i], s2);
                    ag8[i] = hmul2_f16(ag8[i], s28);
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const uint4 xv = xs[(blk * NT + nt) * 32 + lane];
                    mma_16816(acc[nt], ag[0], ag8[0], ag[1], ag8[1], xv.x, xv.y, acc[nt]);
                    mma_16816(acc[nt], ag[2], ag8[2], ag[3], ag8[3], xv.z, xv.w, acc[nt]);
                }
                continue;
            }
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

// Register budget, measured (same GB300, A/B): a single GEMM's short split-K
// items run fastest with the budget set for the CTAs per SM that fit (no
// spills in the per-item path); the grouped launches' long items with the
// compiler's own budget.
template <int NT, int RG, int KW, int STAGES, int G, bool NV = false>
__global__ void __launch_bounds__(GemmCfg<NT, RG, KW, STAGES, NV>::kThreads,
                                  G == 1 ? GemmCfg<NT, RG, KW, STAGES, NV>::kMinBlocks : 0)
    mxfp4_gemm_kernel(const __grid_constant__ ProblemSet<G> S) {
    using C = GemmCfg<NT, RG, KW, STAGES, NV>;
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
            if (pb.sc_from_prep) tma_2d(stage + C::kWBytes, &pb.tm_s, NV ? 2 * kb : kb, n0, bar, pol_w);
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
                    !mbar_wait(empty_bar + 8 * slot, ((it / STAGES) - 1) & 1, S.status, S.wait_ns)) {
                    ok = false;
                    break;
                }
                // (tests only) a stage with no copies and no arrival: its consumers' bounded
                // wait runs out; only stages past the deferred ones, so no copy is left
                if (it == S.skip_stage && blockIdx.x == 0 && it >= STAGES) continue;
                const int kb = R.kb0 + i * kStageBlocks;
                const int nb = min(kStageBlocks, R.kb1 - kb);
                const uint32_t stage = smem_base + slot * C::kStageBytes;
                const uint32_t bar = full_bar + 8 * slot;
                if (G > 1 && i == 0) sh_item[slot] = w;
                mbar_arrive_expect_tx(bar, uint32_t(C::kWBytes + C::kSBytes) +
                                               uint32_t(nb) * NT * kFragBytesPerBlockTile);
                tma_2d(stage, &pb.tm_w, kb * 16, n0, bar, pol_w);
                tma_2d(stage + C::kBoxW, &pb.tm_w, kb * 16 + kBoxBytes, n0, bar, pol_w);
                if (!pb.sc_from_prep) tma_2d(stage + C::kWBytes, &pb.tm_s, NV ? 2 * kb : kb, n0, bar, pol_w);
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
            mbar_wait(full_bar + 8 * (j % STAGES), (j / STAGES) & 1, S.status, S.wait_ns);
        // end of the item stream (after the waits above, which read the
        // slots' current phases): a slot whose barrier completes without copies
        if (G > 1 && ok) {
            const int slot = it % STAGES;
            if (it < STAGES || mbar_wait(empty_bar + 8 * slot, ((it / STAGES) - 1) & 1, S.status, S.wait_ns)) {
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
                if (mbar_wait(full_bar + 8 * slot, (it / STAGES) & 1, S.status, S.wait_ns)) w = sh_item[slot];
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
            if (!mbar_wait(full_bar + 8 * slot, (it / STAGES) & 1, S.status, S.wait_ns)) {
                ok = false;
                break;
            }
            const int nb = min(kStageBlocks, R.kb1 - (R.kb0 + i * kStageBlocks));
            const uint8_t* stage = smem + slot * C::kStageBytes;
            constexpr int kWords = C::kScaleWords / KW;  // scale words (4 scales each) per k-warp
            const uint32_t* s_row = reinterpret_cast<const uint32_t*>(stage + C::kWBytes);
            uint32_t sgw[kWords], sg8w[kWords];
#pragma unroll
            for (int q = 0; q < kWords; ++q) {
                sgw[q] = s_row[(rbase + g) * C::kScaleWords + kw * kWords + q];
                sg8w[q] = s_row[(rbase + g + 8) * C::kScaleWords + kw * kWords + q];
            }
            constexpr int kBlocksPerWarp = kStageBlocks / KW;
            const uint4* xs = reinterpret_cast<const uint4*>(stage + C::kWBytes + C::kSBytes) +
                              kw * kBlocksPerWarp * NT * 32;
            // k-warp kw starts at block kw*16/KW: box (kw*16/KW)/8, chunk pairs from 0
            const uint32_t w_row = smem_base + slot * C::kStageBytes + uint32_t(lrow) * kBoxBytes +
                                   uint32_t((kw * kBlocksPerWarp) / 8) * C::kBoxW;
            const int nbl = nb - kw * kBlocksPerWarp;
            if (nb == kStageBlocks)
                consume_stage<NT, C::kBoxW, KW, true, NV>(acc, w_row, lm, sgw, sg8w, xs, lane, nbl);
            else
                consume_stage<NT, C::kBoxW, KW, false, NV>(acc, w_row, lm, sgw, sg8w, xs, lane, nbl);
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
                if (r < rows) P.y[int64_t(m) * P.N + n0 + r] = NV ? (tile_val(r, m) * P.xun[m]) * P.gscale
                                                                  : tile_val(r, m) * P.xun[m];
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
                        // a single GEMM's tail waits on this sum; the grouped
                        // kernel's main loop is faster as compiled with the
                        // plain loop (same-box A/B)
                        if constexpr (G == 1) {
                            s = sum_partials(P.part + int64_t(R.tile) * M * C::BN + int64_t(m) * C::BN + r,
                                             int64_t(P.ntiles) * M * C::BN, P.nsplit);
                        } else {
                            for (int q = 0; q < P.nsplit; ++q)
                                s += __ldcg(P.part + (int64_t(q) * P.ntiles + R.tile) * M * C::BN +
                                            int64_t(m) * C::BN + r);
                        }
                        P.y[int64_t(m) * P.N + n0 + r] = NV ? (s * P.xun[m]) * P.gscale : s * P.xun[m];
                    }
                }
                if (threadIdx.x == 0) P.counters[R.tile] = 0;  // ready for the next call
            }
        }
    }
}
