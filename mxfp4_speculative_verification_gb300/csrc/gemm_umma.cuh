// Wide-M verify GEMM on sm_103a tensor cores (tcgen05 / UMMA), included by gemm.cu.
//
// For M > 24 candidate positions the legacy mma.sync path runs out of tensor
// throughput before HBM does, so this kernel issues tcgen05.mma (kind::f16,
// fp32 accumulate in tensor memory) with
//   * A = 128 weight rows x 16 k, decoded by CUDA-core warps straight into
//     tensor memory (tcgen05.st): E2M1 -> fp16 by the hardware conversion,
//     times 2^(e_b - e_ref + 13), where e_b is the block's E8M0 exponent and
//     e_ref the largest exponent of that weight row over all of K;
//   * B = the prepared X tile (Npad rows x 512 k, fp16) in shared memory in
//     the 128-byte-swizzled K-major layout, delivered by one bulk copy;
//   * D = 128 x Npad fp32 in tensor memory, double buffered across tiles: a
//     whole 128-row tile accumulates into one D, which is read back once and
//     scaled by 2^(e_ref - 127 - 13).
// A weight w = e2m1 * 2^(e_b - e_ref + 13) is an exact fp16 normal number
// (between 2^-14 and 6 * 2^13) while e_b - e_ref >= -26.  Blocks further
// below their row's maximum are taken out of the MMA (zeros in A) and added
// exactly on the CUDA cores into a second tensor-memory accumulator E, so the
// result is the same for every exponent pattern.
//
// Warps: 0 = TMA producer, 1 = MMA issuer (also owns the TMEM allocation),
// 2 = row-exponent warp (reads each tile's scale rows from global memory one
// tile ahead and publishes e_ref per row), 3..18 = decoders.  A decoder warp
// reaches TMEM lane quadrant warp % 4; the four decoders of a quadrant take
// blocks 4j..4j+3 (j = 0..3) of every 16-block stage.  The j = 0 decoders
// also run the rare exact path and read D back.
//
// Hand-offs: the MMA warp waits once per stage (all 16 decoders arrive on
// the slot's `sready`), then issues the stage's 32 MMAs back to back and
// frees each quarter's A columns with its own commit.  A satisfied mbarrier
// wait costs a few hundred cycles during which the tensor pipe starves, so
// per-stage rather than per-quarter waits matter more than anything else
// in this kernel.

constexpr int kUBN = 128;                    // weight rows per tile (MMA M)
constexpr int kUDecodeWarps = 16;
constexpr int kUFirstDecoder = 3;
constexpr int kUThreads = 32 * (kUFirstDecoder + kUDecodeWarps);
constexpr uint32_t kUTmemCols = 512;
constexpr uint32_t kUASetCols = 64;          // one A set: a quarter stage, 4 blocks x 16 columns
constexpr int kUWindow = 26;                 // binades below the row maximum kept in fp16
constexpr int kUBias = 13;                   // A = e2m1 * 2^(e_b - e_ref + kUBias)

// Tensor-memory map.  The A ring takes what D leaves: 7 quarter-stage sets
// (1.75 stages) for N_pad <= 32, 6 for 48, 5 for 64.  The exact-path
// accumulator E lives in shared memory where it fits (N_pad <= 48) and in
// the last 64 columns otherwise.
template <int NPAD>
struct UTmem {
    static constexpr bool kESmem = NPAD <= 48;
    static constexpr int kASets = NPAD <= 32 ? 7 : (NPAD <= 48 ? 6 : 5);
    static constexpr uint32_t kDCol0 = uint32_t(kASets) * kUASetCols;
    static constexpr uint32_t kDStride = NPAD <= 32 ? 32 : 64;
    static constexpr uint32_t kECol = 448;  // used only when !kESmem
    static_assert(kDCol0 + 2 * kDStride <= (kESmem ? kUTmemCols : kECol), "TMEM map");
    static_assert(kESmem || kECol + 64 <= kUTmemCols, "TMEM map");
};

template <int NPAD, int STAGES>
struct UCfg {
    using T = UTmem<NPAD>;
    static constexpr int kBoxW = kUBN * kBoxBytes;               // 16 KB nibble box
    static constexpr int kWBytes = 2 * kBoxW;
    static constexpr int kSBytes = kUBN * 16;
    static constexpr int kXBytes = NPAD * 1024;                   // NPAD rows x 512 k fp16
    static constexpr int kStageBytes = kWBytes + kSBytes + kXBytes;
    static constexpr int kMaskOffset = STAGES * kStageBytes;      // uint8 [STAGES][4][128]
    static constexpr int kErefOffset = kMaskOffset + STAGES * 4 * kUBN;  // int32 [2][128]
    static constexpr int kLowOffset = kErefOffset + 2 * kUBN * 4;        // int32 [2]: tile has low blocks
    static constexpr int kEPitch = NPAD + 1;                              // floats per row of E
    static constexpr int kEOffset = kLowOffset + 16;                      // fp32 [128][NPAD + 1] if in smem
    static constexpr int kBarOffset = kEOffset + (T::kESmem ? kUBN * kEPitch * 4 : 0);
    // full[S], empty[S], maskfull[S], sready[S], afree[5], dready[2], dfree[2],
    // efull[2], efree[2], fin
    static constexpr int kNumBars = 4 * STAGES + T::kASets + 9;
    static constexpr int kMiscOffset = kBarOffset + kNumBars * 8;
    static constexpr int kSmemBytes = kMiscOffset + 16 + 1024;
    static_assert(kStageBytes % 1024 == 0, "swizzled tiles need 1 KB alignment");
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
    static_assert(NPAD % 16 == 0 && NPAD >= 16 && NPAD <= 64, "MMA N");
    static_assert(kBarOffset % 8 == 0, "mbarrier alignment");
};

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}
// D[128 x N] (+)= A[128 x 16, TMEM] * B[N x 16, smem]^T
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// 16 columns of this warp's 32 lanes
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]));
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// One lane of a converged warp (the lowest active one) gets true.
__device__ __forceinline__ bool elect_one() {
    uint32_t pred = 0;
    asm volatile(
        "{\n .reg .pred P;\n elect.sync _|P, 0xffffffff;\n selp.b32 %0, 1, 0, P;\n}\n"
        : "=r"(pred));
    return pred != 0;
}

// Shared-memory descriptor of a K-major, 128-byte-swizzled operand tile
// (rows of 128 bytes, 8-row groups 1024 bytes apart).
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_addr) {
    return (uint64_t((smem_addr >> 4) & 0x3FFFu)) | (uint64_t(1) << 16) |
           (uint64_t(1024 >> 4) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// Instruction descriptor: fp16 x fp16 -> fp32, both K-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t umma_idesc_f16(int n) {
    return (1u << 4) | (uint32_t(n >> 3) << 17) | (uint32_t(kUBN >> 4) << 24);
}

// fp16x2 holding 2^p in both halves, p in [-14, 15] (a normal fp16 power of two).
__device__ __forceinline__ uint32_t f16x2_pow2_normal(int p) {
    const uint32_t h = uint32_t(p + 15) << 10;
    return h | (h << 16);
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ float f16_lo(uint32_t v) {
    return __half2float(__ushort_as_half(uint16_t(v & 0xFFFFu)));
}
__device__ __forceinline__ float f16_hi(uint32_t v) {
    return __half2float(__ushort_as_half(uint16_t(v >> 16)));
}

// Byte-wise maximum of acc and w after NaN scales (255) and the bytes at or
// above `valid` (the bytes of w that belong to the row, clamped to 0..4)
// are replaced by 0.
__device__ __forceinline__ uint32_t scale_word_max(uint32_t acc, uint32_t w, int valid) {
    const uint32_t keep = valid >= 4 ? 0xFFFFFFFFu : (valid <= 0 ? 0u : (1u << (8 * valid)) - 1u);
    const uint32_t nan = __vcmpeq4(w, 0xFFFFFFFFu);
    return __vmaxu4(acc, w & ~nan & keep);
}

// Byte-wise minimum of acc and w over the bytes below `valid`.  NaN scales
// (255) never lower the minimum.
__device__ __forceinline__ uint32_t scale_word_min(uint32_t acc, uint32_t w, int valid) {
    const uint32_t keep = valid >= 4 ? 0xFFFFFFFFu : (valid <= 0 ? 0u : (1u << (8 * valid)) - 1u);
    return __vminu4(acc, w | ~keep);
}

// Decode one 32-k block of a weight row (16 bytes of nibbles) into 16 fp16x2.
__device__ __forceinline__ void decode_block(uint4 nib, uint32_t (&v)[16]) {
    e2m1x8_to_f16x2x4(nib.x, v[0], v[1], v[2], v[3]);
    e2m1x8_to_f16x2x4(nib.y, v[4], v[5], v[6], v[7]);
    e2m1x8_to_f16x2x4(nib.z, v[8], v[9], v[10], v[11]);
    e2m1x8_to_f16x2x4(nib.w, v[12], v[13], v[14], v[15]);
}

// Exact CUDA-core contribution of one block that lies outside the fp16
// window, for candidate rows c0..c0+15:
// ea[m - c0] += 2^(e-127) * sum_k v_k * x[m][k].
template <int NPAD>
__device__ __forceinline__ void exact_block16(float (&ea)[16], const uint32_t (&v)[16], int e,
                                              const uint8_t* xtile, int blk, int c0, int M) {
    const float s = pow2f_exact(e - 127);
    const uint8_t* chunk = xtile + (blk >> 1) * (NPAD * 128);
#pragma unroll
    for (int mm = 0; mm < 16; ++mm) {
        const int m = c0 + mm;
        if (m < M) {
            const uint8_t* row = chunk + m * 128;
            float sum = 0.f;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const int k0 = (blk & 1) * 32 + 2 * c;  // k within the 64-k chunk
                const int u = k0 >> 3, eo = k0 & 7;
                const uint32_t xx =
                    *reinterpret_cast<const uint32_t*>(row + ((u ^ (m & 7)) << 4) + eo * 2);
                sum = fmaf(f16_lo(v[c]), f16_lo(xx), sum);
                sum = fmaf(f16_hi(v[c]), f16_hi(xx), sum);
            }
            ea[mm] = fmaf(sum, s, ea[mm]);
        }
    }
}

template <int NPAD, int STAGES, int G>
__global__ void __launch_bounds__(kUThreads, 1)
    mxfp4_gemm_umma_kernel(const __grid_constant__ ProblemSet<G> S) {
    using C = UCfg<NPAD, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_base & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    const uint32_t sbase = raw_base + pad;
    const uint32_t bars = sbase + C::kBarOffset;
    auto full_b = [&](int s) { return bars + 8u * s; };
    auto empty_b = [&](int s) { return bars + 8u * (STAGES + s); };
    // j = 1..3 -> j = 0 hand-off of the out-of-window masks of one stage slot;
    // its next phase needs the slot refilled, so it never runs ahead of its waiter
    auto maskfull_b = [&](int s) { return bars + 8u * (2 * STAGES + s); };
    // all four quarters of the stage in a slot are decoded (one wait per stage for
    // the MMA warp: each wait costs a few hundred cycles of tensor-pipe idle time)
    auto sready_b = [&](int s) { return bars + 8u * (3 * STAGES + s); };
    // quarter stage t = 4 * it + j decodes into A set t % 5, freed by the MMA's
    // commit (u-th use: parity (t / 5) & 1)
    auto afree_b = [&](int a) { return bars + 8u * (4 * STAGES + a); };
    constexpr int kASets = C::T::kASets;
    constexpr int kB2 = 4 * STAGES + kASets;
    auto dready_b = [&](int d) { return bars + 8u * (kB2 + d); };
    auto dfree_b = [&](int d) { return bars + 8u * (kB2 + 2 + d); };
    auto efull_b = [&](int d) { return bars + 8u * (kB2 + 4 + d); };
    auto efree_b = [&](int d) { return bars + 8u * (kB2 + 6 + d); };
    const uint32_t fin_b = bars + 8u * (kB2 + 8);
    uint32_t* tbase_ptr = reinterpret_cast<uint32_t*>(smem + C::kMiscOffset);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOffset + 4);
    uint8_t* masks = smem + C::kMaskOffset;
    int* eref_s = reinterpret_cast<int*>(smem + C::kErefOffset);
    volatile int* tlow_s = reinterpret_cast<volatile int*>(smem + C::kLowOffset);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_b(s), 1);
            mbar_init(empty_b(s), 1 + kUDecodeWarps);  // MMA commit + every decoder warp
            mbar_init(maskfull_b(s), 12);              // the j = 1..3 decoders
            mbar_init(sready_b(s), kUDecodeWarps);
        }
        for (int a = 0; a < kASets; ++a) mbar_init(afree_b(a), 1);
        for (int d = 0; d < 2; ++d) {
            mbar_init(dready_b(d), 1);
            mbar_init(dfree_b(d), 4);
            mbar_init(efull_b(d), 32);
            mbar_init(efree_b(d), kUDecodeWarps);
        }
        mbar_init(fin_b, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(tbase_ptr), kUTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_trigger();
    const uint32_t tbase = *tbase_ptr;
    const int M = S.M;

    // Bounded wait that gives up for the whole CTA after the first timeout.
    // Every lane polls: on a completed phase that returns in about half the
    // time of one lane polling and broadcasting the result.
    auto wait = [&](uint32_t bar, uint32_t parity) -> bool {
        if (*abort_flag) return false;
        if (mbar_wait(bar, parity, S.status)) return true;
        *abort_flag = 1;
        return false;
    };

    if (warp == 0) {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            int def_slot[STAGES], def_st[STAGES], def_pi[STAGES];
            int ndef = 0;
            bool waited = false;
            auto issue_x = [&](int slot, int st, int pi) {
                bulk_g2s(sbase + slot * C::kStageBytes + C::kWBytes + C::kSBytes,
                         S.p[pi].xf + int64_t(st) * (NPAD * 512), uint32_t(C::kXBytes),
                         full_b(slot), pol_x);
            };
            auto wait_pdl = [&]() {
                pdl_wait();
                waited = true;
                for (int d = 0; d < ndef; ++d) issue_x(def_slot[d], def_st[d], def_pi[d]);
                ndef = 0;
            };
            int it = 0, last_pi = -1;
            bool ok = true;
            for (int w = blockIdx.x; ok && w < S.items; w += gridDim.x) {
                const int pi = find_problem(S, w);
                const Problem& pb = S.p[pi];
                if (pi != last_pi) {
                    prefetch_tmap(&pb.tm_w);
                    prefetch_tmap(&pb.tm_s);
                    last_pi = pi;
                }
                // scales realigned by the preparation kernel are read after it
                if (pb.sc_from_prep && !waited) wait_pdl();
                const ItemRange R = item_range(pb, w - pb.item_begin);
                const int n0 = R.tile * kUBN;
                for (int i = 0; i < R.nst; ++i, ++it) {
                    const int slot = it % STAGES;
                    if (it >= STAGES && !wait(empty_b(slot), ((it / STAGES) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    const int kb = R.kb0 + i * kStageBlocks;
                    const uint32_t stage = sbase + slot * C::kStageBytes;
                    mbar_arrive_expect_tx(full_b(slot), uint32_t(C::kWBytes + C::kSBytes + C::kXBytes));
                    tma_2d(stage, &pb.tm_w, kb * 16, n0, full_b(slot), pol_w);
                    tma_2d(stage + C::kBoxW, &pb.tm_w, kb * 16 + kBoxBytes, n0, full_b(slot), pol_w);
                    tma_2d(stage + C::kWBytes, &pb.tm_s, kb, n0, full_b(slot), pol_w);
                    const int st = kb / kStageBlocks;  // stage index of the prepared X
                    if (waited) {
                        issue_x(slot, st, pi);
                    } else {
                        def_slot[ndef] = slot;
                        def_st[ndef] = st;
                        def_pi[ndef] = pi;
                        if (++ndef == STAGES) wait_pdl();
                    }
                }
            }
            if (!waited) wait_pdl();
            for (int j = max(0, it - STAGES); j < it; ++j)
                mbar_wait(full_b(j % STAGES), (j / STAGES) & 1, S.status);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer
        // The whole warp walks the schedule (so its state stays warp-uniform);
        // one elected lane issues the MMAs and their commits.
        constexpr uint32_t idesc = umma_idesc_f16(NPAD);
        int it = 0, tc = 0;
        bool ok = true;
        for (int w = blockIdx.x; ok && w < S.items; w += gridDim.x, ++tc) {
            const Problem& pb = S.p[find_problem(S, w)];
            const ItemRange R = item_range(pb, w - pb.item_begin);
            const int db = tc & 1;
            if (tc >= 2 && !wait(dfree_b(db), ((tc >> 1) - 1) & 1)) { ok = false; break; }
            const uint32_t d_t = tbase + C::T::kDCol0 + C::T::kDStride * db;
            for (int i = 0; ok && i < R.nst; ++i, ++it) {
                const int slot = it % STAGES;
                const int nb = min(kStageBlocks, R.kb1 - (R.kb0 + i * kStageBlocks));
                if (!wait(full_b(slot), (it / STAGES) & 1)) { ok = false; break; }
                if (!wait(sready_b(slot), (it / STAGES) & 1)) { ok = false; break; }
                tc_fence_after();
                // descriptor of the stage's X tile; block b, k-step jj starts
                // (b >> 1) * NPAD * 128 + ((b & 1) * 2 + jj) * 32 bytes further
                const uint64_t xd = umma_desc_sw128(sbase + slot * C::kStageBytes + C::kWBytes + C::kSBytes);
                if (elect_one()) {
                    for (int j = 0; j < 4; ++j) {
                        const int t = 4 * it + j;
                        const int set = t % kASets;
                        const uint32_t a0 = tbase + kUASetCols * set;
                        const uint64_t xq = xd + uint64_t((j * 2 * NPAD * 128) >> 4);
                        const int nbq = min(4, nb - 4 * j);
                        if (nbq == 4) {
#pragma unroll
                            for (int bb = 0; bb < 4; ++bb)
#pragma unroll
                                for (int jj = 0; jj < 2; ++jj)
                                    umma_f16_ts(d_t, a0 + 16u * bb + 8u * jj,
                                                xq + uint64_t((((bb >> 1) * NPAD * 128) + ((bb & 1) * 2 + jj) * 32) >> 4),
                                                idesc, (i | j | bb | jj) != 0);
                        } else {
                            for (int bb = 0; bb < nbq; ++bb)
                                for (int jj = 0; jj < 2; ++jj)
                                    umma_f16_ts(d_t, a0 + 16u * bb + 8u * jj,
                                                xq + uint64_t((((bb >> 1) * NPAD * 128) + ((bb & 1) * 2 + jj) * 32) >> 4),
                                                idesc, (i | j | bb | jj) != 0);
                        }
                        tc_commit(afree_b(set));
                    }
                    tc_commit(empty_b(slot));
                }
                __syncwarp();
            }
            if (ok && elect_one()) tc_commit(dready_b(db));
            __syncwarp();
        }
        // every issued MMA has completed before the allocation is released
        if (elect_one()) tc_commit(fin_b);
        __syncwarp();
        mbar_wait(fin_b, 0, S.status);
    } else if (warp == 2) {
        // ---------------------------------------------- row exponents e_ref
        bool waited = false;
        int tc = 0;
        for (int w = blockIdx.x; w < S.items; w += gridDim.x, ++tc) {
            const int es = tc & 1;
            if (tc >= 2 && !wait(efree_b(es), ((tc >> 1) - 1) & 1)) break;
            const Problem& pb = S.p[find_problem(S, w)];
            if (pb.sc_from_prep && !waited) {
                pdl_wait();
                waited = true;
            }
            const ItemRange R = item_range(pb, w - pb.item_begin);
            const int64_t n0 = int64_t(R.tile) * kUBN;
            const int nchunk = (pb.nblk + 15) >> 4;
            const int tail = pb.nblk - 16 * (nchunk - 1);  // bytes of the row in its last chunk
            // pull the next tile's scale rows into L2 now, so that reading them a
            // tile from now waits on L2 rather than HBM
            const int wn = w + int(gridDim.x);
            if (wn < S.items) {
                const Problem& pn = S.p[find_problem(S, wn)];
                const int64_t nn0 = int64_t(item_range(pn, wn - pn.item_begin).tile) * kUBN;
                const int lines = int((pn.nblk + 127) >> 7);
                for (int rr = 0; rr < 4; ++rr) {
                    const int64_t n = nn0 + lane + 32 * rr;
                    if (n < pn.N)
                        for (int l = 0; l < lines; ++l)
                            asm volatile("prefetch.global.L2 [%0];" ::"l"(pn.sc + n * pn.sc_pitch + 128 * l));
                }
            }
            bool low = false;  // some row has a block below its fp16 window
#pragma unroll 1
            for (int rr = 0; rr < 4; ++rr) {
                const int r = lane + 32 * rr;
                uint32_t mx = 0, mn = 0xFFFFFFFFu;
                if (n0 + r < pb.N) {
                    const uint4* row = reinterpret_cast<const uint4*>(pb.sc + (n0 + r) * pb.sc_pitch);
#pragma unroll 4
                    for (int c = 0; c < nchunk - 1; ++c) {
                        const uint4 v = __ldg(row + c);
                        mx = scale_word_max(mx, v.x, 4);
                        mx = scale_word_max(mx, v.y, 4);
                        mx = scale_word_max(mx, v.z, 4);
                        mx = scale_word_max(mx, v.w, 4);
                        mn = __vminu4(__vminu4(mn, v.x), __vminu4(v.y, __vminu4(v.z, v.w)));
                    }
                    const uint4 v = __ldg(row + nchunk - 1);
                    mx = scale_word_max(mx, v.x, tail);
                    mx = scale_word_max(mx, v.y, tail - 4);
                    mx = scale_word_max(mx, v.z, tail - 8);
                    mx = scale_word_max(mx, v.w, tail - 12);
                    mn = scale_word_min(mn, v.x, tail);
                    mn = scale_word_min(mn, v.y, tail - 4);
                    mn = scale_word_min(mn, v.z, tail - 8);
                    mn = scale_word_min(mn, v.w, tail - 12);
                }
                mx = __vmaxu4(mx, mx >> 16);
                mx = __vmaxu4(mx, mx >> 8);
                mn = __vminu4(mn, mn >> 16);
                mn = __vminu4(mn, mn >> 8);
                eref_s[es * kUBN + r] = int(mx & 0xFFu);
                low |= int(mn & 0xFFu) < int(mx & 0xFFu) - kUWindow;
            }
            low = __any_sync(0xffffffffu, low);
            if (lane == 0) tlow_s[es] = low ? 1 : 0;
            __syncwarp();
            mbar_arrive(efull_b(es));
        }
    } else {
        // ------------------------------------------------------- decoders
        const int q = warp & 3;                              // TMEM lane quadrant
        const int j = (warp - kUFirstDecoder) >> 2;          // blocks 4j..4j+3 of a stage
        const int r = 32 * q + lane;                         // weight row within the tile
        const uint32_t lane_addr = uint32_t(32 * q) << 16;
        // the exact-path accumulator E of this thread's row: 16 columns at a time
        float* erow = reinterpret_cast<float*>(smem + C::kEOffset) + r * C::kEPitch;
        auto e_load16 = [&](int c0, uint32_t (&ev)[16]) {
            if constexpr (C::T::kESmem) {
#pragma unroll
                for (int c = 0; c < 16; ++c) ev[c] = c0 + c < NPAD ? __float_as_uint(erow[c0 + c]) : 0u;
            } else {
                tmem_ld16(tbase + lane_addr + C::T::kECol + c0, ev);
            }
        };
        auto e_store16 = [&](int c0, const uint32_t (&ev)[16]) {
            if constexpr (C::T::kESmem) {
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    if (c0 + c < NPAD) erow[c0 + c] = __uint_as_float(ev[c]);
            } else {
                tmem_st16(tbase + lane_addr + C::T::kECol + c0, ev);
            }
        };
        bool waited_pdl = false;
        bool e_used = false;                                 // E holds exact-path sums (j = 0)
        int it = 0, tc = 0;
        bool ok = true;
        // the tile whose D is still to be read back (j = 0)
        int pd_tc = -1, pd_eref = 0, pd_rows = 0;
        const Problem* pd_pb = nullptr;
        int64_t pd_n0 = 0;
        auto drain = [&]() -> bool {
            const int db = pd_tc & 1;
            if (!wait(dready_b(db), (pd_tc >> 1) & 1)) return false;
            tc_fence_after();
            if (!waited_pdl) {
                pdl_wait();  // Y and xun belong to the preceding kernels until now
                waited_pdl = true;
            }
            // y = (D * 2^(e_ref - 127 - 13) + E) * xun, the power of two applied in
            // at most two exact steps
            const float s1 = pd_eref >= 14 ? 1.f : 0x1p-13f;
            const float s2 = pow2f_exact(pd_eref >= 14 ? pd_eref - 127 - kUBias : pd_eref - 127);
            float* yrow = pd_pb->y + pd_n0 + r;
            const float* xun = pd_pb->xun;
            const int64_t N = pd_pb->N;
#pragma unroll 1
            for (int c0 = 0; c0 < NPAD; c0 += 16) {
                uint32_t dv[16], ev[16];
                tmem_ld16(tbase + lane_addr + C::T::kDCol0 + C::T::kDStride * db + c0, dv);
                if (e_used) e_load16(c0, ev);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const int m = c0 + c;
                    const float e = e_used ? __uint_as_float(ev[c]) : 0.f;
                    if (m < M && r < pd_rows)
                        yrow[int64_t(m) * N] = fmaf(__uint_as_float(dv[c]) * s1, s2, e) * xun[m];
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(dfree_b(db));
                mbar_arrive(efree_b(pd_tc & 1));
            }
            e_used = false;
            pd_tc = -1;
            return true;
        };
        for (int w = blockIdx.x; ok && w < S.items; w += gridDim.x, ++tc) {
            const Problem& pb = S.p[find_problem(S, w)];
            const ItemRange R = item_range(pb, w - pb.item_begin);
            const int64_t n0 = int64_t(R.tile) * kUBN;
            const int rows = int(pb.N - n0 < int64_t(kUBN) ? pb.N - n0 : int64_t(kUBN));
            const int es = tc & 1;
            if (!wait(efull_b(es), (tc >> 1) & 1)) { ok = false; break; }
            const int eref = eref_s[es * kUBN + r];
            // without blocks below the fp16 window anywhere in the tile, the j = 0
            // warps neither wait for the others' masks nor run the exact path
            const bool tile_low = tlow_s[es] != 0;
            for (int i = 0; i < R.nst; ++i, ++it) {
                const int slot = it % STAGES;
                const int nb = min(kStageBlocks, R.kb1 - (R.kb0 + i * kStageBlocks));
                if (!wait(full_b(slot), (it / STAGES) & 1)) { ok = false; break; }
                const uint8_t* stage = smem + slot * C::kStageBytes;
                const int t = 4 * it + j;
                const int set = t % kASets;
                if (t >= kASets && !wait(afree_b(set), ((t / kASets) - 1) & 1)) { ok = false; break; }
                // per-block fp16 multipliers 2^(e - e_ref + 13): 0 takes a block out of
                // the MMA (beyond the stage's blocks, or below the fp16 window), NaN
                // for a NaN scale
                const uint32_t sw = *reinterpret_cast<const uint32_t*>(stage + C::kWBytes + r * 16 + 4 * j);
                uint32_t mul[4];
                uint32_t om = 0;
#pragma unroll
                for (int bb = 0; bb < 4; ++bb) {
                    const int e = int((sw >> (8 * bb)) & 0xFFu);
                    const int d = e - eref;
                    const bool live = 4 * j + bb < nb;
                    const bool low = live && e != 255 && d < -kUWindow;
                    om |= low ? (1u << bb) : 0u;
                    mul[bb] = !live || low ? 0u : (e == 255 ? 0x7E007E00u : f16x2_pow2_normal(d + kUBias));
                }
#pragma unroll
                for (int bb = 0; bb < 4; ++bb) {
                    const int b = 4 * j + bb;
                    uint32_t v[16];
                    const uint4 nib = *reinterpret_cast<const uint4*>(
                        stage + (b >> 3) * C::kBoxW + r * kBoxBytes + (((b & 7) ^ (r & 7)) << 4));
                    decode_block(nib, v);
#pragma unroll
                    for (int c = 0; c < 16; ++c) v[c] = hmul2_u32(v[c], mul[bb]);
                    tmem_st16(tbase + lane_addr + kUASetCols * set + 16u * bb, v);
                }
                if (j > 0 && tile_low) masks[(slot * 4 + j) * kUBN + r] = uint8_t(om);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(sready_b(slot));
                    if (j > 0) {
                        mbar_arrive(maskfull_b(slot));
                        mbar_arrive(empty_b(slot));
                    }
                }
                if (j == 0) {
                    // the previous tile's D is complete once this tile's first quarter is out
                    if (pd_tc >= 0 && !drain()) { ok = false; break; }
                    // blocks below the fp16 window (rare), all 16 of the stage: exact on
                    // the CUDA cores while the stage is still resident, summed into E.
                    // (The j = 1..3 warps arrive on maskfull at every use of the slot;
                    // waiting only in flagged tiles keeps the phases aligned, since no
                    // arrival of a slot's next use precedes this warp's empty arrival.)
                    if (tile_low && !wait(maskfull_b(slot), (it / STAGES) & 1)) { ok = false; break; }
                    const uint32_t om16 =
                        !tile_low ? 0u
                                  : om | (uint32_t(masks[(slot * 4 + 1) * kUBN + r]) << 4) |
                                        (uint32_t(masks[(slot * 4 + 2) * kUBN + r]) << 8) |
                                        (uint32_t(masks[(slot * 4 + 3) * kUBN + r]) << 12);
                    if (__any_sync(0xffffffffu, om16 != 0)) {
                        const uint4 srow = *reinterpret_cast<const uint4*>(stage + C::kWBytes + r * 16);
                        const uint32_t sws[4] = {srow.x, srow.y, srow.z, srow.w};
                        const uint8_t* xtile = stage + C::kWBytes + C::kSBytes;
                        if (!e_used) {
                            uint32_t z[16];
#pragma unroll
                            for (int c = 0; c < 16; ++c) z[c] = 0u;
#pragma unroll
                            for (int c0 = 0; c0 < NPAD; c0 += 16) e_store16(c0, z);
                            tmem_wait_st();
                            e_used = true;
                        }
#pragma unroll 1
                        for (int c0 = 0; c0 < NPAD; c0 += 16) {
                            uint32_t ev[16];
                            e_load16(c0, ev);
                            tmem_wait_ld();
                            float ea[16];
#pragma unroll
                            for (int c = 0; c < 16; ++c) ea[c] = __uint_as_float(ev[c]);
#pragma unroll 1
                            for (int b = 0; b < 16; ++b) {
                                if (!((om16 >> b) & 1u)) continue;
                                uint32_t v[16];
                                const uint4 nib = *reinterpret_cast<const uint4*>(
                                    stage + (b >> 3) * C::kBoxW + r * kBoxBytes + (((b & 7) ^ (r & 7)) << 4));
                                decode_block(nib, v);
                                const int e = int((sws[b >> 2] >> (8 * (b & 3))) & 0xFFu);
                                exact_block16<NPAD>(ea, v, e, xtile, b, c0, M);
                            }
                            __syncwarp();
#pragma unroll
                            for (int c = 0; c < 16; ++c) ev[c] = __float_as_uint(ea[c]);
                            e_store16(c0, ev);
                        }
                        tmem_wait_st();
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(empty_b(slot));
                }
            }
            if (!ok) break;
            if (j > 0) {
                __syncwarp();
                if (lane == 0) mbar_arrive(efree_b(es));
            } else {
                pd_tc = tc;
                pd_eref = eref;
                pd_pb = &pb;
                pd_n0 = n0;
                pd_rows = rows;
            }
        }
        if (ok && j == 0 && pd_tc >= 0) drain();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tbase, kUTmemCols);
}
