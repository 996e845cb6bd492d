// Block-scaled verify GEMM on sm_103a tensor cores, included by gemm.cu.
//
// tcgen05.mma.kind::mxf8f6f4.block_scale multiplies E2M1 weights by E4M3
// activations, each 32-k block scaled by one UE8M0 factor per weight row
// (A) and per activation row (B), and accumulates in fp32 in tensor memory.
// That is the MX-FP4 product of "Module 11. Speculative Decoding and
// Quantization" §12 (E2M1 elements, one power-of-two scale per 32-element
// block) done by the tensor core itself: no weight is ever decoded.
//   * A = 128 weight rows x 256 k per stage.  The MMA reads E2M1 codes from
//     a padded shared-memory layout (each 16 codes = 8 bytes, then 8 unused
//     bytes); TMA writes that layout from the packed bytes in HBM (the
//     16U4_ALIGN16B type).  Each request of that type covers 64 bytes of a
//     row, and one 2-D box per 128 k capped a whole GPU near 3 TB/s (measured),
//     so one 3-D box carries both 128-k chunks of a stage: 5.3 TB/s for the
//     stream alone.  The A scale factors are the weight's own E8M0 bytes,
//     unchanged.
//   * B = X as two E4M3 terms: x = t1 * 2^e1 + t2 * 2^e2 per 32-k block,
//     e1 set by the block's largest |x| and e2 by the largest residual
//     (the preparation kernel).  Every bf16 value whose block maximum is
//     within 2^16 of it is represented exactly, the rest to 16 bits.  The
//     terms are stacked as B rows (row m = t1 of X row m, row Npad + m = t2),
//     so one MMA of N = 2 Npad per 32-k block reads A from shared memory
//     once, and Y[m] = D[m] + D[Npad + m].
//   * D = 128 x 2 Npad fp32 in tensor memory, double buffered across tiles.
//
// Scale factors in tensor memory (pinned on this GPU by a one-CTA probe of
// every placement against a host reference): the MMA reads row m's A factor
// at lane m, column base + m / 32, byte 0 (factor id 0), and B column n's
// factor at lane 32 * (m / 32) + n % 32 of the sub-partition computing row m,
// column base + n / 32.  Each 32-k block gets a group of 4 columns (factor
// addresses stay 4-column aligned): lane m holds its A factor in all 4, and
// every lane quadrant holds the same copy of B's factors, column base + c
// for B columns n = lane + 32 c.  Every tcgen05.st starts at a column that
// is a multiple of its width.
//
// Warps: 0 = weight producer (one 3-D TMA box per stage), 1 = MMA issuer
// (and tensor-memory owner), 2..5 = scale-factor warps (one per lane
// quadrant: write both operands' factors into tensor memory, flag NaN
// scales), 6..9 = epilogue warps (tensor memory -> Y, or a split-K partial
// tile and its reduction), 10 = X producer (bulk copies of the prepared X
// terms).  A stage slot holds a stage's weights, X terms and (in tensor
// memory) factors; its full barrier completes when both copies have landed
// and the factors are written, so the MMA warp waits once and commits once
// per stage (each wait and commit of that single issuing thread costs the
// tensor pipe idle time).

constexpr int kBsRows = 128;                 // weight rows per tile (MMA M)
constexpr int kBsStageBlocks = 8;            // 32-k blocks per stage (256 k)
constexpr int kBsAChunk = kBsRows * 128;     // one 128-k chunk of A in the padded layout
constexpr int kBsAStage = 2 * kBsAChunk;     // padded A of one stage (32 KB)
constexpr int kBsATx = kBsRows * 128;        // its packed global bytes (the transaction count)
constexpr int kBsMaxNpad = 64;               // X rows per pass at most
constexpr int kBsFirstEpi = 6;
constexpr int kBsXWarp = 10;
constexpr int kBsThreads = 32 * 11;
constexpr uint32_t kBsTmemCols = 512;
constexpr int kBsMaxRing = 8;
constexpr int kBsPfStages = 10;              // L2 prefetch distance of the weights (MXS_GEMM_BS_PF)

// X rows a pass pads to: 32 or 64 (MMA N = 64 or 128, the widths this
// kernel's block-scaled MMA has been validated at on this GPU).
__host__ __device__ constexpr int bs_npad(int m) { return m <= 32 ? 32 : 64; }
// Prepared X, per 256-k stage: B rows [2 chunks of 128 k][2 Npad rows][128 B]
// (K-major, 16-byte units swizzled by row % 8; rows 0..Npad-1 = t1, then
// t2); after all stages, their scale bytes [stage][2 Npad][8 blocks].
__host__ __device__ constexpr int bs_bstage_bytes(int npad) { return 512 * npad; }
__host__ __device__ constexpr int bs_sfbstage_bytes(int npad) { return 16 * npad; }
// One stage slot: padded A, then B.
__host__ __device__ constexpr int bs_slot_bytes(int npad) { return kBsAStage + bs_bstage_bytes(npad); }
// Tensor-memory columns: D buffer 0 at column 0 (2 Npad wide), then one
// factor slot of 64 columns per stage slot (A: 8 blocks x 4, B: 8 blocks x 4),
// then D buffer 1 at a multiple of 2 Npad (a power of two).
constexpr int kBsSfCols = 64;
constexpr int kBsSfbCol = 32;  // B's factors within a slot
__host__ __device__ constexpr int bs_sf0(int npad) { return 2 * npad; }
__host__ __device__ constexpr int bs_d1(int npad, int ring) {
    return (bs_sf0(npad) + ring * kBsSfCols + 2 * npad - 1) / (2 * npad) * (2 * npad);
}
__host__ __device__ constexpr int bs_tmem_need(int npad, int ring) { return bs_d1(npad, ring) + 2 * npad; }
// shared memory beyond the ring: barriers, NaN flags, TMEM base, abort flag
constexpr int kBsMiscBytes = 8 * 64 + 2 * kBsRows + 64;
__host__ __device__ constexpr int bs_smem_bytes(int npad, int ring) {
    return ring * bs_slot_bytes(npad) + kBsMiscBytes + 1024;
}
// Stage slots (48 or 64 KB each) that fit.
__host__ __device__ constexpr int bs_ring(int npad) { return npad <= 32 ? 4 : 3; }

struct BsItem {
    int tile, split, kb0, kb1, nst;
};

__device__ __forceinline__ BsItem bs_item(const Problem& P, int w) {
    BsItem r;
    r.tile = w % P.ntiles;
    r.split = w / P.ntiles;
    r.kb0 = r.split * P.stages_per_split * kBsStageBlocks;
    r.kb1 = min(P.nblk, r.kb0 + P.stages_per_split * kBsStageBlocks);
    r.nst = r.kb1 > r.kb0 ? (r.kb1 - r.kb0 + kBsStageBlocks - 1) / kBsStageBlocks : 0;
    return r;
}

// Position in this CTA's stream of stages: item w (round robin over the
// CTAs), stage i of it.  The fields of the item's GEMM that each stage needs
// are copied into registers once per item: reading them from the launch
// table on every stage costs a dependent parameter load each.
template <int G>
struct BsCursor {
    int w, i;
    int pi;                 // problem of item w (valid while w < items)
    BsItem R;
    const uint8_t* sc;      // its scale rows, pitch sc_pitch
    int64_t sc_pitch;
    int64_t N;
    const uint8_t* xf;      // its prepared X
    int nst_all;            // stages of its whole K
    bool w8;                // scale rows readable 8 bytes at a time
    __device__ __forceinline__ void load(const ProblemSet<G>& S) {
        if (w < S.items) {
            pi = find_problem(S, w);
            const Problem& P = S.p[pi];
            R = bs_item(P, w - P.item_begin);
            sc = P.sc;
            sc_pitch = P.sc_pitch;
            N = P.N;
            xf = reinterpret_cast<const uint8_t*>(P.xf);
            nst_all = (P.nblk + kBsStageBlocks - 1) / kBsStageBlocks;
            w8 = ((sc_pitch | int64_t(reinterpret_cast<uintptr_t>(sc))) & 7) == 0;
        }
    }
    __device__ __forceinline__ void start(const ProblemSet<G>& S) {
        w = int(blockIdx.x);
        i = 0;
        load(S);
    }
    __device__ __forceinline__ void next(const ProblemSet<G>& S) {
        if (w >= S.items) return;
        if (++i >= R.nst) {
            i = 0;
            w += int(gridDim.x);
            load(S);
        }
    }
    __device__ __forceinline__ bool valid(const ProblemSet<G>& S) const { return w < S.items; }
    __device__ __forceinline__ int kb() const { return R.kb0 + i * kBsStageBlocks; }
    __device__ __forceinline__ int nb() const { return min(kBsStageBlocks, R.kb1 - kb()); }
};

// D[128 x N] (+)= A[128 x 32] * B[N x 32]^T with one UE8M0 factor per row of
// A and of B for the 32-k block (instruction descriptor `idesc`).
__device__ __forceinline__ void umma_mxf8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%5], [%6], p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

// Instruction descriptor: A E2M1 (5), B E4M3 (0), UE8M0 factors (bit 23),
// both K-major, M = 128, N = n, factor ids 0.
__host__ __device__ constexpr uint32_t bs_idesc(int n) {
    return (5u << 7) | (0u << 10) | (uint32_t(n >> 3) << 17) | (1u << 23) | (uint32_t(kBsRows >> 4) << 24);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
        "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
        "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
        "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31]));
}

// The 8 scale bytes of blocks kb .. kb+7 at `p` (fewer at the end of K;
// missing ones read as 0), as two little-endian words.
__device__ __forceinline__ uint2 bs_load8(const uint8_t* p, int nb, bool w8) {
    if (nb == kBsStageBlocks && w8) return __ldg(reinterpret_cast<const uint2*>(p));
    uint32_t lo = 0, hi = 0;
    for (int j = 0; j < nb; ++j) {
        const uint32_t b = __ldg(p + j);
        if (j < 4) lo |= b << (8 * j);
        else hi |= b << (8 * (j - 4));
    }
    return make_uint2(lo, hi);
}

__device__ __forceinline__ bool has_byte_ff(uint32_t w) { return __vcmpeq4(w, 0xFFFFFFFFu) != 0; }

// The factors one stage-warp thread writes for one stage: its weight row's
// 8 bytes, and those of B rows lane + 32 c (c = 0..3).
struct BsFactors {
    uint2 a;
    uint2 b[4];
};

template <int G>
__device__ __forceinline__ BsFactors bs_load_factors(const ProblemSet<G>& S, const BsCursor<G>& c, int r,
                                                     int lane, int npad) {
    BsFactors f;
    f.a = make_uint2(0u, 0u);
#pragma unroll
    for (int j = 0; j < 4; ++j) f.b[j] = make_uint2(0u, 0u);
    if (!c.valid(S)) return f;
    const int kb = c.kb(), nb = c.nb();
    const int64_t n = int64_t(c.R.tile) * kBsRows + r;
    if (n < c.N) f.a = bs_load8(c.sc + n * c.sc_pitch + kb, nb, c.w8);
    // X-term scales: after the stages' B rows
    const uint8_t* sfb = c.xf + int64_t(c.nst_all) * bs_bstage_bytes(npad) +
                         int64_t(kb / kBsStageBlocks) * bs_sfbstage_bytes(npad);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int row = lane + 32 * j;
        if (row < 2 * npad) f.b[j] = __ldg(reinterpret_cast<const uint2*>(sfb + row * 8));
    }
    return f;
}

// One stage's factors into factor slot `sf` (a TMEM address with this warp's
// lane quadrant, 32-column aligned): block j of A in columns sf + 4j ..
// sf + 4j + 3 (this thread's row's byte in all four), block j of B in
// columns sf + 32 + 4j + c (B column lane + 32 c, the same in every quadrant).
__device__ __forceinline__ void bs_write_factors(uint32_t sf, const BsFactors& f) {
    {
        uint32_t v[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t b = ((j < 4 ? f.a.x : f.a.y) >> (8 * (j & 3))) & 0xFFu;
            v[4 * j] = v[4 * j + 1] = v[4 * j + 2] = v[4 * j + 3] = b;
        }
        tmem_st32(sf, v);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // blocks 4h .. 4h + 3
        uint32_t v[16];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
#pragma unroll
            for (int c = 0; c < 4; ++c) v[4 * jj + c] = ((h ? f.b[c].y : f.b[c].x) >> (8 * jj)) & 0xFFu;
        tmem_st16(sf + uint32_t(kBsSfbCol + 16 * h), v);
    }
}

template <int G>
__global__ void __launch_bounds__(kBsThreads, 1)
    mxfp4_gemm_bs_kernel(const __grid_constant__ ProblemSet<G> S) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_base & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    const uint32_t sbase = raw_base + pad;
    const int M = S.M;
    const int npad = bs_npad(M);
    const int R = S.ring;
    const int bbytes = bs_bstage_bytes(npad);
    const int slot_bytes = bs_slot_bytes(npad);
    const uint32_t d1col = uint32_t(bs_d1(npad, R));
    const int misc = R * slot_bytes;
    const uint32_t bars = sbase + misc;
    // a stage slot is full once both producers' bytes have landed and the four
    // scale-factor warps have written its factors: the MMA warp waits once
    auto full_b = [&](int c) { return bars + 8u * c; };
    auto empty_b = [&](int c) { return bars + 8u * (kBsMaxRing + c); };
    constexpr int kB2 = 2 * kBsMaxRing;
    auto dready_b = [&](int d) { return bars + 8u * (kB2 + d); };
    auto dfree_b = [&](int d) { return bars + 8u * (kB2 + 2 + d); };
    auto flags_b = [&](int d) { return bars + 8u * (kB2 + 4 + d); };
    const uint32_t fin_b = bars + 8u * (kB2 + 6);
    static_assert(kB2 + 7 <= 64, "barrier area");
    uint8_t* nanflags = smem + misc + 8 * 64;                       // [2][128]
    uint32_t* tbase_ptr = reinterpret_cast<uint32_t*>(smem + misc + 8 * 64 + 2 * kBsRows);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + misc + 8 * 64 + 2 * kBsRows + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int c = 0; c < R; ++c) {
            mbar_init(full_b(c), 2 + 4);  // two producers (with their bytes) + four scale-factor warps
            mbar_init(empty_b(c), 1);     // the MMA commit
        }
        for (int d = 0; d < 2; ++d) {
            mbar_init(dready_b(d), 1);
            mbar_init(dfree_b(d), 4);
            mbar_init(flags_b(d), 4);
        }
        mbar_init(fin_b, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(tbase_ptr), kBsTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_trigger();
    const uint32_t tbase = *tbase_ptr;
    const uint32_t sf0 = tbase + uint32_t(bs_sf0(npad));

    // every wait of this kernel sleeps rather than spins: the scale-factor warps
    // share their schedulers with the epilogue and producer warps, which wait
    // for most of a tile
    auto wait = [&](uint32_t bar, uint32_t parity) -> bool {
        if (*abort_flag) return false;
        if (mbar_wait_sleep(bar, parity, S.status)) return true;
        *abort_flag = 1;
        return false;
    };

    if (warp == 0 || warp == kBsXWarp) {
        // ------------------------------------ producers (weights / prepared X)
        if (lane == 0) {
            const bool wprod = warp == 0;
            const uint64_t pol = wprod ? policy_evict_first() : policy_evict_last();
            if (!wprod) pdl_wait();  // the prepared X belongs to the preparation kernel until now
            BsCursor<G> cur, pf;
            cur.start(S);
            pf.start(S);
            // weights: each stage's boxes prefetched into L2 S.pf_stages stages before
            // they are loaded, so that the ring waits on L2 rather than HBM latency
            auto prefetch = [&]() {
                if (!pf.valid(S)) return;
                const Problem& pp = S.p[pf.pi];
                const bool two = pf.nb() > 4;
                asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                                 reinterpret_cast<uint64_t>(two ? &pp.tm_w : &pp.tm_s)),
                             "r"(0), "r"(pf.R.tile * kBsRows), "r"(pf.kb() / 4)
                             : "memory");
                pf.next(S);
            };
            if (wprod)
                for (int j = 0; j < S.pf_stages; ++j) prefetch();
            int it = 0, last_pi = -1;
            for (; cur.valid(S); cur.next(S), ++it) {
                const int c = it % R;
                if (wprod && S.pf_stages > 0) prefetch();
                if (it >= R && !wait(empty_b(c), ((it / R) - 1) & 1)) break;
                const uint32_t slot = sbase + uint32_t(c * slot_bytes);
                if (wprod) {
                    const Problem& pb = S.p[cur.pi];
                    if (cur.pi != last_pi) {
                        prefetch_tmap(&pb.tm_w);
                        prefetch_tmap(&pb.tm_s);
                        last_pi = cur.pi;
                    }
                    // both 128-k chunks in one request (tm_w), or the last chunk of an
                    // odd count alone (tm_s)
                    const bool two = cur.nb() > 4;
                    mbar_arrive_expect_tx(full_b(c), uint32_t(two ? kBsATx : kBsATx / 2));
                    asm volatile(
                        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(slot),
                        "l"(reinterpret_cast<uint64_t>(two ? &pb.tm_w : &pb.tm_s)), "r"(0),
                        "r"(cur.R.tile * kBsRows), "r"(cur.kb() / 4), "r"(full_b(c)), "l"(pol)
                        : "memory");
                } else {
                    mbar_arrive_expect_tx(full_b(c), uint32_t(bbytes));
                    bulk_g2s(slot + kBsAStage, cur.xf + int64_t(cur.kb() / kBsStageBlocks) * bbytes,
                             uint32_t(bbytes), full_b(c), pol);
                }
            }
            // never leave a copy in flight
            for (int j = max(0, it - R); j < it; ++j) mbar_wait_sleep(full_b(j % R), (j / R) & 1, S.status);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer
        const uint32_t idesc = bs_idesc(2 * npad);
        int it = 0, tc = 0;
        bool ok = true;
        for (int w = int(blockIdx.x); ok && w < S.items; w += int(gridDim.x), ++tc) {
            const Problem& pb = S.p[find_problem(S, w)];
            const BsItem RI = bs_item(pb, w - pb.item_begin);
            const int db = tc & 1;
            if (tc >= 2 && !wait(dfree_b(db), ((tc >> 1) - 1) & 1)) { ok = false; break; }
            const uint32_t d_t = tbase + (db ? d1col : 0u);
            for (int i = 0; ok && i < RI.nst; ++i, ++it) {
                const int c = it % R;
                const int nb = min(kBsStageBlocks, RI.kb1 - (RI.kb0 + i * kBsStageBlocks));
                if (!wait(full_b(c), (it / R) & 1)) { ok = false; break; }
                tc_fence_after();
                if (lane == 0) {
                    // descriptors advance by 32 bytes per block within a 128-k chunk
                    // (2 in their 16-byte address field) and by a chunk after four
                    const uint32_t slot = sbase + uint32_t(c * slot_bytes);
                    const uint64_t ad0 = umma_desc_sw128(slot);
                    const uint64_t bd0 = umma_desc_sw128(slot + kBsAStage);
                    const uint32_t sfa = sf0 + uint32_t(kBsSfCols * c);
#pragma unroll
                    for (int kb = 0; kb < kBsStageBlocks; ++kb) {
                        if (kb < nb)
                            umma_mxf8f6f4(d_t, ad0 + uint64_t(((kb >> 2) * kBsAChunk + (kb & 3) * 32) >> 4),
                                          bd0 + uint64_t(((kb >> 2) * (2 * npad * 128) + (kb & 3) * 32) >> 4),
                                          idesc, sfa + uint32_t(4 * kb), sfa + uint32_t(kBsSfbCol + 4 * kb),
                                          (i | kb) != 0);
                    }
                    tc_commit(empty_b(c));
                }
                __syncwarp();
            }
            if (ok && lane == 0) tc_commit(dready_b(db));
            __syncwarp();
        }
        // every issued MMA has completed before the allocation is released
        if (lane == 0) tc_commit(fin_b);
        __syncwarp();
        mbar_wait_sleep(fin_b, 0, S.status);
    } else if (warp < kBsFirstEpi) {
        // ------------------------------------------------ scale-factor warps
        const int q = warp & 3;
        const int r = 32 * q + lane;
        const uint32_t lane_addr = uint32_t(32 * q) << 16;
        // The factors of a stage are loaded three stages before they are
        // written: three buffers used in turn (the loop is unrolled by three),
        // so that no register copy waits for a load.  X's factors are written
        // by the preparation kernel: read only after it has finished.
        pdl_wait();
        BsCursor<G> cur, ld, pf;
        cur.start(S);
        ld.start(S);
        pf.start(S);
        BsFactors fa = bs_load_factors(S, ld, r, lane, npad);
        ld.next(S);
        BsFactors fb = bs_load_factors(S, ld, r, lane, npad);
        ld.next(S);
        BsFactors fc = bs_load_factors(S, ld, r, lane, npad);
        ld.next(S);
        for (int j = 0; j < 8; ++j) pf.next(S);
        int it = 0, tc = 0;
        bool nan = false;
        // one stage: write its factors into the slot's columns once the MMA is done with them
        auto stage = [&](const BsFactors& f) -> bool {
            const int c = it % R;
            // the weight scales 8 stages ahead into L2, one prefetch per 32-byte sector
            if (pf.valid(S) && (pf.kb() & 31) == 0) {
                const int64_t n = int64_t(pf.R.tile) * kBsRows + r;
                if (n < pf.N) asm volatile("prefetch.global.L2 [%0];" ::"l"(pf.sc + n * pf.sc_pitch + pf.kb()));
            }
            pf.next(S);
            nan |= has_byte_ff(f.a.x) || has_byte_ff(f.a.y);
            if (it >= R && !wait(empty_b(c), ((it / R) - 1) & 1)) return false;
            bs_write_factors(sf0 + uint32_t(kBsSfCols * c) + lane_addr, f);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(full_b(c));
            ++it;
            if (cur.i == cur.R.nst - 1) {
                // the tile's NaN-scale flags, once the epilogue is done with the slot's previous tile
                const int db = tc & 1;
                if (tc >= 2 && !wait(dfree_b(db), ((tc >> 1) - 1) & 1)) return false;
                nanflags[db * kBsRows + r] = nan ? 1 : 0;
                __syncwarp();
                if (lane == 0) mbar_arrive(flags_b(db));
                nan = false;
                ++tc;
            }
            cur.next(S);
            return true;
        };
        while (cur.valid(S)) {
            if (!stage(fa)) break;
            fa = bs_load_factors(S, ld, r, lane, npad);
            ld.next(S);
            if (!cur.valid(S)) break;
            if (!stage(fb)) break;
            fb = bs_load_factors(S, ld, r, lane, npad);
            ld.next(S);
            if (!cur.valid(S)) break;
            if (!stage(fc)) break;
            fc = bs_load_factors(S, ld, r, lane, npad);
            ld.next(S);
        }
    } else {
        // ------------------------------------------------------- epilogue
        const int q = warp & 3;
        const int r = 32 * q + lane;
        const uint32_t lane_addr = uint32_t(32 * q) << 16;
        bool waited_pdl = false;
        int tc = 0;
        for (int w = int(blockIdx.x); w < S.items; w += int(gridDim.x), ++tc) {
            const Problem& pb = S.p[find_problem(S, w)];
            const int wl = w - pb.item_begin;
            const BsItem R = bs_item(pb, wl);
            const int64_t n0 = int64_t(R.tile) * kBsRows;
            const int rows = int(pb.N - n0 < int64_t(kBsRows) ? pb.N - n0 : int64_t(kBsRows));
            const int db = tc & 1;
            if (!wait(dready_b(db), (tc >> 1) & 1)) break;
            if (!wait(flags_b(db), (tc >> 1) & 1)) break;
            tc_fence_after();
            if (!waited_pdl) {
                pdl_wait();  // Y, xun, partials and counters belong to the preceding kernels until now
                waited_pdl = true;
            }
            const bool nan = nanflags[db * kBsRows + r] != 0;
            const float* xun = pb.xun;
            const int64_t N = pb.N;
            float* mine = pb.part + int64_t(wl) * M * kBsRows;
            const uint32_t dcol = tbase + lane_addr + (db ? d1col : 0u);
#pragma unroll 1
            for (int c0 = 0; c0 < npad; c0 += 16) {
                uint32_t d1[16], d2[16];
                tmem_ld16(dcol + uint32_t(c0), d1);
                tmem_ld16(dcol + uint32_t(npad + c0), d2);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const int m = c0 + c;
                    if (m < M) {
                        const float v = nan ? __int_as_float(0x7FC00000)
                                            : __uint_as_float(d1[c]) + __uint_as_float(d2[c]);
                        if (pb.nsplit == 1) {
                            if (r < rows) pb.y[int64_t(m) * N + n0 + r] = v * xun[m];
                        } else {
                            __stcg(mine + int64_t(m) * kBsRows + r, v);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dfree_b(db));
            if (pb.nsplit > 1) {
                // each warp's 32 rows of the tile are counted apart: the warp that
                // brings the last split of them sums all splits in split order
                __threadfence();
                __syncwarp();
                int last = 0;
                if (lane == 0) last = atomicAdd(pb.counters + 4 * R.tile + q, 1) == pb.nsplit - 1;
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
                    __threadfence();
                    if (r < rows)
                        for (int m = 0; m < M; ++m) {
                            float s = 0.f;
                            for (int sp = 0; sp < pb.nsplit; ++sp)
                                s += __ldcg(pb.part + (int64_t(sp) * pb.ntiles + R.tile) * M * kBsRows +
                                            int64_t(m) * kBsRows + r);
                            pb.y[int64_t(m) * N + n0 + r] = s * xun[m];
                        }
                    if (lane == 0) pb.counters[4 * R.tile + q] = 0;  // ready for the next call
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tbase, kBsTmemCols);
}
