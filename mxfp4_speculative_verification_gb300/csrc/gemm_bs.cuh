// Block-scaled verify GEMM on sm_103a tensor cores, included by gemm.cu.
//
// tcgen05.mma with .block_scale multiplies E2M1 weights by a low-precision
// image of X, each 32-k block scaled by one UE8M0 factor per weight row (A)
// and per X term row (B), and accumulates in fp32 in tensor memory.  That is
// the MX-FP4 product of "Module 11. Speculative Decoding and Quantization"
// §12 (E2M1 elements, one power-of-two scale per 32-element block) done by
// the tensor core itself: no weight is ever decoded.  Two kinds:
//   * kind::mxf8f6f4 (KIND 0, passes of 33..64 rows): B = X as two E4M3
//     terms per 32-k block, x = t1 * 2^e1 + t2 * 2^e2, exact for every bf16
//     element within 2^16 of its block maximum.  The MMA reads E2M1 codes
//     from a padded shared-memory layout (16 codes = 8 bytes, then 8 unused
//     bytes), which TMA writes from the packed bytes (the 16U4_ALIGN16B
//     type): 32 KB of shared memory per 16 KB of weights.
//   * kind::mxf4 (KIND 1, passes of up to 32 rows): A = the packed E2M1
//     bytes as they are (16 KB per 16 KB, plain 128-byte-swizzled TMA boxes),
//     B = X as six E2M1 terms per 32-k block, each with its own UE8M0 scale
//     (the largest residual maps into (3, 6]).  Six terms carry X to about
//     1e-7 of its block maximum on normal data; the bound for any block is
//     the residual after six terms, at most max|x| / 4^6.
//   * kind::mxf4nvf4 (KIND 2, NVFP4 weights, passes of up to 64 rows): A =
//     the packed E2M1 bytes, each 16-k block scaled by its E4M3 byte read as
//     UE4M3 (scale_vec::4X: one 32-bit factor cell per MMA of 64 k); B = X
//     as four E2M1 terms per 16-k block, each with its own UE4M3 factor (the
//     smallest at or above the residual's maximum / 6).  A negative weight
//     scale is folded into its block's codes (sign bits flipped in shared
//     memory before the MMA reads them); the tensor's FP32 scale multiplies
//     Y in the epilogue.  Four terms carry a bf16 row to ~1e-5 of its
//     maximum (rows are first scaled by a power of two into [2^10, 2^11),
//     inside the UE4M3 range).
//   * kind::mxf4 in W4A4 form (KIND 3, passes of up to 256 rows): X itself
//     quantised to MX-FP4 by the pack rule (one E2M1 term per element, one
//     UE8M0 factor per 32-k block; rows below 1 scaled up by a power of
//     two first, which the rule commutes with), so the product is that of
//     the quantised X ("Module 11 ...", §12, W4A4); N = the pass's rows,
//     so W is streamed once for up to 256 rows.
//   The terms are stacked as B rows (row t * Npad + m = term t of X row m),
//   so one MMA of N = T * Npad reads A from shared memory once, and
//   Y[m] = sum over t of D[t * Npad + m].  Shared memory per stage is what
//   bounds the bytes in flight, hence the mxf4 kind where its six terms fit.
//
// Scale factors (pinned on this GPU by one-CTA probes against a host double
// reference): one 32-bit tensor-memory cell holds the factors of four
// consecutive 32-k blocks (byte j = block 4g + j); the MMA's factor id picks
// the byte (mxf8f6f4: one block per MMA) or the byte pair (mxf4,
// scale_vec::2X: two blocks per MMA).  A's factor of weight row m is read at
// lane m, column base + m / 32, and B column n's at lane 32 q + n % 32 of
// every lane quadrant q, column base + n / 32.  The scale-factor warps write
// both with tcgen05.st, each into its own lane quadrant: the weight scales
// from a TMA box that comes with the weights (16 bytes x 128 rows), X's
// cells from the stage's prepared X (laid out for them by the preparation
// kernel).
//
// What bounds a stage (measured with per-stage clocks on this GPU): the one
// MMA-issuing thread spends ~70-90 cycles per tcgen05 instruction, and a
// stage of 16 KB of weights must take no more than ~750 cycles to keep pace
// with HBM, so that thread issues only the stage's MMAs and one commit: the
// factors reach tensor memory through the scale-factor warps instead of
// tcgen05.cp, and its loop runs on one lane.  Loading the weight scales
// with per-thread 8-byte loads cost ~40 % of the stream (as many memory
// requests as the weights themselves); the TMA box costs ~10 %.
//
// Warps: 0 = weight producer (per 256-k stage one TMA box of weights and
// one of their scales), 1 = MMA issuer (and tensor-memory owner), 2..5 =
// scale-factor warps (one per lane quadrant: factors into tensor memory,
// flag NaN scales), 6..9 = epilogue warps (tensor memory -> Y, or a split-K
// partial tile and its reduction), 10 = X producer (one bulk copy of the
// stage's prepared X and its factors).  A stage slot's full barrier
// completes when both copies have landed; its factor barrier when the four
// scale-factor warps have written the factors (which they do after the full
// barrier), so the MMA thread waits on the factor barrier alone.

constexpr int kBsRows = 128;                 // weight rows per tile (MMA M)
constexpr int kBsStageBlocks = 8;            // 32-k blocks per stage (256 k)
constexpr int kBsAChunk = kBsRows * 128;     // mxf8f6f4: one 128-k chunk of padded A
constexpr int kBsATx = kBsRows * 128;        // packed global bytes of a stage's A
constexpr int kBsMaxNpad = 64;               // X rows per pass at most
constexpr int kBsF4Terms = 6;                // E2M1 terms of X (mxf4 kind)
constexpr int kBsNvTerms = 4;                // E2M1 terms of X (mxf4nvf4 kind)
constexpr int kBsFirstEpi = 6;
constexpr int kBsXWarp = 10;
constexpr int kBsThreads = 32 * 11;
constexpr uint32_t kBsTmemCols = 512;
constexpr int kBsMaxRing = 8;
constexpr int kBsScBytes = kBsRows * 16;     // TMA box of weight scales: 16 blocks x 128 rows
constexpr int kBsCopyBytes = 512;            // one group x 128 columns of X's factor cells
constexpr int kBsF4MaxRows = 32;             // the mxf4 kind takes passes of at most this many rows
constexpr int kBsW4MaxRows = 256;            // W4A4 (X as one E2M1 term): MMA N up to 256

// X rows a pass pads to (multiples of 16 keep every term row group's swizzle
// and tensor-memory columns aligned).
__host__ __device__ constexpr int bs_npad(int kind, int m) {
    return kind == 3   ? (m + 15) / 16 * 16
           : kind == 2 ? (m <= 16 ? 16 : (m <= 32 ? 32 : 64))
                       : (kind ? (m <= 16 ? 16 : 32) : (m <= 32 ? 32 : 64));
}
// X rows a pass of this kind takes at most
__host__ __device__ constexpr int bs_max_rows(int kind) { return kind == 3 ? kBsW4MaxRows : (kind == 1 ? 32 : 64); }
// One D buffer in tensor memory instead of two (the next tile's MMAs wait for
// the epilogue): NVFP4 passes of 33..64 rows, whose N = 4 x 64 = 256 columns
// leave no room for a second buffer beside the factor slots, and W4A4
// passes of more than 192 rows.
__host__ __device__ constexpr bool bs_single_d(int kind, int npad) {
    return (kind == 2 && npad == 64) || (kind == 3 && npad > 192);
}
__host__ __device__ constexpr int bs_terms(int kind) {
    return kind == 3 ? 1 : (kind == 2 ? kBsNvTerms : (kind ? kBsF4Terms : 2));
}
// factor groups per 256-k stage: one per MMA of 64 k (NVFP4), else per 4 blocks of 32 k
__host__ __device__ constexpr int bs_groups(int kind) { return kind == 2 ? 4 : 2; }
// MMA N: the term rows of B
__host__ __device__ constexpr int bs_ncols(int kind, int npad) { return bs_terms(kind) * npad; }
// A of one stage in shared memory (padded for mxf8f6f4)
__host__ __device__ constexpr int bs_a_bytes(int kind) { return kind ? kBsRows * 128 : 2 * kBsRows * 128; }
// 128-column parts of B's factor cells per group
__host__ __device__ constexpr int bs_sfb_copies(int kind, int npad) { return (bs_ncols(kind, npad) + 127) / 128; }
// Prepared X, per 256-k stage: B rows (K-major, 16-byte units swizzled by
// row % 8; mxf8f6f4: [2 chunks of 128 k][N rows][128 B], mxf4: [N rows][128 B]),
// then B's factors: [group g][copy h][32 rows][4 cells], cell c of row l =
// the 4 factor bytes of B column 128 h + 32 c + l for blocks 4 g .. 4 g + 3
// (32-k blocks; 16-k blocks for NVFP4, one group per MMA).
__host__ __device__ constexpr int bs_brows_bytes(int kind, int npad) { return bs_ncols(kind, npad) * (kind ? 128 : 256); }
__host__ __device__ constexpr int bs_sfb_bytes(int kind, int npad) {
    return bs_groups(kind) * bs_sfb_copies(kind, npad) * kBsCopyBytes;
}
__host__ __device__ constexpr int bs_bstage_bytes(int kind, int npad) {
    return bs_brows_bytes(kind, npad) + bs_sfb_bytes(kind, npad);
}
// One stage slot: A, the stage's prepared X (B rows and factors), the weight scales.
__host__ __device__ constexpr int bs_slot_bytes(int kind, int npad) {
    return bs_a_bytes(kind) + bs_bstage_bytes(kind, npad) + kBsScBytes;
}
// Tensor-memory columns: D buffer 0 at column 0 (N wide), then one factor
// slot per stage slot (A: groups x 4 columns, then B: groups x 4 columns per
// copy; every factor address a multiple of 4 columns), then D buffer 1 at the
// next multiple of 64.
__host__ __device__ constexpr int bs_sf_cols(int kind, int npad) {
    return 4 * bs_groups(kind) * (1 + bs_sfb_copies(kind, npad));
}
__host__ __device__ constexpr int bs_sf0(int kind, int npad) { return bs_ncols(kind, npad); }
__host__ __device__ constexpr int bs_d1(int kind, int npad, int ring) {
    return bs_single_d(kind, npad) ? 0 : (bs_sf0(kind, npad) + ring * bs_sf_cols(kind, npad) + 63) / 64 * 64;
}
__host__ __device__ constexpr int bs_tmem_need(int kind, int npad, int ring) {
    return bs_single_d(kind, npad) ? bs_sf0(kind, npad) + ring * bs_sf_cols(kind, npad)
                                   : bs_d1(kind, npad, ring) + bs_ncols(kind, npad);
}
// shared memory beyond the ring: barriers, NaN flags, TMEM base, abort flag
constexpr int kBsMiscBytes = 8 * 64 + 2 * kBsRows + 64;
// Output staging of single-GEMM launches (Y written by TMA tensor stores):
// per epilogue warp two buffers of 16 rows x 32 fp32 columns.
constexpr int kBsYStageBytes = 4 * 2 * 16 * 32 * 4;
// Offset of the output staging (1024-aligned, after the barriers and flags).
__host__ __device__ constexpr int bs_ystage_off(int kind, int npad, int ring) {
    return (ring * bs_slot_bytes(kind, npad) + kBsMiscBytes + 1023) / 1024 * 1024;
}
__host__ __device__ constexpr int bs_smem_bytes(int kind, int npad, int ring, int ybytes = 0) {
    return ybytes ? bs_ystage_off(kind, npad, ring) + ybytes + 1024 : ring * bs_slot_bytes(kind, npad) + kBsMiscBytes + 1024;
}
constexpr int kBsSmemAttr = 232448;  // dynamic shared memory the kernel may ask for
// Stage slots: as many as shared and tensor memory hold (at most kBsMaxRing).
__host__ __device__ constexpr int bs_ring(int kind, int npad, int ybytes = 0) {
    int r = kBsMaxRing;
    while (r > 2 &&
           (bs_smem_bytes(kind, npad, r, ybytes) > kBsSmemAttr || bs_tmem_need(kind, npad, r) > int(kBsTmemCols)))
        --r;
    return r;
}

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

// D[128 x N] (+)= A[128 x K] * B[N x K]^T, one factor per row and 32-k block
// (instruction descriptor `idesc`; K = 32 for mxf8f6f4, 64 for mxf4).
template <int KIND>
__device__ __forceinline__ void umma_bs(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    if constexpr (KIND == 2)
        asm volatile(
            "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
            " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n}\n" ::"r"(
                d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
            : "memory");
    else if constexpr (KIND == 0)
        asm volatile(
            "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
            " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%5], [%6], p;\n}\n" ::"r"(
                d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
            : "memory");
    else
        asm volatile(
            "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
            " tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n}\n" ::"r"(
                d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
            : "memory");
}

// Instruction descriptor: M = 128, N = n, both K-major; mxf8f6f4: A E2M1
// (5), B E4M3 (0); mxf4 and mxf4nvf4: A and B E2M1 (1).  Factors UE8M0 (bit
// 23 set), or UE4M3 for mxf4nvf4 (clear).  The factor ids (A: bits 29-30, B:
// bits 4-5) are or-ed in per MMA by bs_sfid (always 0 for mxf4nvf4).
__host__ __device__ constexpr uint32_t bs_idesc(int kind, int n) {
    return (kind ? ((1u << 7) | (1u << 10)) : (5u << 7)) | (uint32_t(n >> 3) << 17) | (kind == 2 ? 0u : (1u << 23)) |
           (uint32_t(kBsRows >> 4) << 24);
}
__device__ __forceinline__ uint32_t bs_sfid(uint32_t j) { return (j << 29) | (j << 4); }

__device__ __forceinline__ bool has_byte_ff(uint32_t w) { return __vcmpeq4(w, 0xFFFFFFFFu) != 0; }

// TMA tensor store of a shared-memory box to global memory (bulk-group
// completion), and the group operations of the issuing thread.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int c0, int c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// all but the newest group have finished reading their shared memory
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// every group has completed (its writes performed)
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Wait for this thread's tensor-memory loads, naming the registers the last
// one writes: the compiler then keeps every read of them after the wait.
__device__ __forceinline__ void tmem_wait_ld_into(uint32_t (&v)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]), "+r"(v[7]),
                   "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]), "+r"(v[14]),
                   "+r"(v[15])
                 :
                 : "memory");
}

__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(a), "r"(b),
                 "r"(c), "r"(d)
                 : "memory");
}

template <int G, int KIND>
__global__ void __launch_bounds__(kBsThreads, 1)
    mxfp4_gemm_bs_kernel(const __grid_constant__ ProblemSet<G> S) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_base & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    const uint32_t sbase = raw_base + pad;
    const int M = S.M;
    const int npad = bs_npad(KIND, M);
    const int T = bs_terms(KIND);
    const int N = bs_ncols(KIND, npad);
    const int copies = bs_sfb_copies(KIND, npad);
    const int R = S.ring;
    const int abytes = bs_a_bytes(KIND);
    const int brows = bs_brows_bytes(KIND, npad);
    const int bbytes = bs_bstage_bytes(KIND, npad);
    const int slot_bytes = bs_slot_bytes(KIND, npad);
    const uint32_t sfcols = uint32_t(bs_sf_cols(KIND, npad));
    const uint32_t d1col = uint32_t(bs_d1(KIND, npad, R));
    const int misc = R * slot_bytes;
    const uint32_t bars = sbase + misc;
    // a stage slot is full once both producers' bytes have landed, and its
    // factors are ready once the four scale-factor warps have written them
    auto full_b = [&](int c) { return bars + 8u * c; };
    auto empty_b = [&](int c) { return bars + 8u * (kBsMaxRing + c); };
    auto sfok_b = [&](int c) { return bars + 8u * (2 * kBsMaxRing + c); };
    constexpr int kB2 = 3 * kBsMaxRing;
    auto dready_b = [&](int d) { return bars + 8u * (kB2 + d); };
    auto dfree_b = [&](int d) { return bars + 8u * (kB2 + 2 + d); };
    auto flags_b = [&](int d) { return bars + 8u * (kB2 + 4 + d); };
    const uint32_t fin_b = bars + 8u * (kB2 + 6);
    static_assert(kB2 + 7 <= 64, "barrier area");
    uint8_t* nanflags = smem + misc + 8 * 64;                       // [2][128]
    constexpr int kYB = G == 1 ? kBsYStageBytes : 0;  // output staging (single-GEMM launches)
    float* ystage = reinterpret_cast<float*>(smem + bs_ystage_off(KIND, npad, R));
    uint32_t* tbase_ptr = reinterpret_cast<uint32_t*>(smem + misc + 8 * 64 + 2 * kBsRows);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + misc + 8 * 64 + 2 * kBsRows + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int c = 0; c < R; ++c) {
            mbar_init(full_b(c), 2);      // two producers (with their bytes)
            mbar_init(sfok_b(c), 4);      // four scale-factor warps
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
            BsCursor<G> cur;
            cur.start(S);
            int it = 0, last_pi = -1;
            bool waited_pdl = !wprod;
            for (; cur.valid(S); cur.next(S), ++it) {
                const int c = it % R;
                if (it >= R && !wait(empty_b(c), ((it / R) - 1) & 1)) break;
                const uint32_t slot = sbase + uint32_t(c * slot_bytes);
                if (wprod) {
                    const Problem& pb = S.p[cur.pi];
                    if (cur.pi != last_pi) {
                        prefetch_tmap(&pb.tm_w);
                        prefetch_tmap(&pb.tm_s);
                        last_pi = cur.pi;
                        if (pb.sc_from_prep && !waited_pdl) {
                            pdl_wait();  // scales realigned by the preparation kernel of this call
                            waited_pdl = true;
                        }
                    }
                    // the weights' scales: the 16-byte column of 16 blocks holding this stage's 8
                    // (NVFP4: the stage's own 16 bytes, one per 16 k)
                    mbar_arrive_expect_tx(full_b(c), uint32_t(kBsATx + kBsScBytes));
                    tma_2d(slot + uint32_t(abytes + bbytes), &pb.tm_s, KIND == 2 ? 2 * cur.kb() : cur.kb() & ~15,
                           cur.R.tile * kBsRows, full_b(c), pol);
                    if constexpr (KIND == 0) {
                        // both 128-k chunks of the stage (a chunk beyond K reads as zero codes)
                        asm volatile(
                            "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                            ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(slot),
                            "l"(reinterpret_cast<uint64_t>(&pb.tm_w)), "r"(0),
                            "r"(cur.R.tile * kBsRows), "r"(cur.kb() / 4), "r"(full_b(c)), "l"(pol)
                            : "memory");
                    } else {
                        // one 128-byte x 128-row box (bytes beyond K / 2 read as zero codes)
                        tma_2d(slot, &pb.tm_w, cur.kb() * 16, cur.R.tile * kBsRows, full_b(c), pol);
                    }
                } else {
                    mbar_arrive_expect_tx(full_b(c), uint32_t(bbytes));
                    bulk_g2s(slot + uint32_t(abytes), cur.xf + int64_t(cur.kb() / kBsStageBlocks) * bbytes,
                             uint32_t(bbytes), full_b(c), pol);
                }
            }
            // never leave a copy in flight
            for (int j = max(0, it - R); j < it; ++j) mbar_wait_sleep(full_b(j % R), (j / R) & 1, S.status);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer
        // one lane: a warp-wide loop costs the tensor pipe a few hundred
        // cycles of every stage in convergence and slot arithmetic
        if (lane == 0) {
            const uint32_t idesc = bs_idesc(KIND, N);
            const uint32_t sf0c = tbase + uint32_t(bs_sf0(KIND, npad));
            int tc = 0, c = 0;
            uint32_t ph = 0;  // parity of slot c's current use
            bool ok = true;
            for (int w = int(blockIdx.x); ok && w < S.items; w += int(gridDim.x), ++tc) {
                const Problem& pb = S.p[find_problem(S, w)];
                const BsItem RI = bs_item(pb, w - pb.item_begin);
                const int db = tc & 1;
                // D of tile tc - 2 (two buffers) or tc - 1 (one) has been read out
                if (bs_single_d(KIND, npad)) {
                    if (tc >= 1 && !wait(dfree_b((tc - 1) & 1), ((tc - 1) >> 1) & 1)) { ok = false; break; }
                } else if (tc >= 2 && !wait(dfree_b(db), ((tc >> 1) - 1) & 1)) {
                    ok = false;
                    break;
                }
                const uint32_t d_t = tbase + (db ? d1col : 0u);
                for (int i = 0; i < RI.nst; ++i) {
                    const int nb = min(kBsStageBlocks, RI.kb1 - (RI.kb0 + i * kBsStageBlocks));
                    // the factors are written after the stage's bytes landed: their barrier covers both
                    if (!mbar_try_wait(sfok_b(c), ph) && !wait(sfok_b(c), ph)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t slot = sbase + uint32_t(c * slot_bytes);
                    const uint64_t ad0 = umma_desc_sw128(slot);
                    const uint64_t bd0 = umma_desc_sw128(slot + uint32_t(abytes));
                    const uint32_t tsfa = sf0c + sfcols * uint32_t(c);
                    const uint32_t tsfb = tsfa + uint32_t(4 * bs_groups(KIND));
                    if constexpr (KIND == 2) {
                        // four MMAs of 64 k, each with its own factor cells (4 x 16 k)
#pragma unroll
                        for (int j = 0; j < kBsStageBlocks / 2; ++j)
                            if (2 * j < nb)
                                umma_bs<2>(d_t, ad0 + uint64_t((j * 32) >> 4), bd0 + uint64_t((j * 32) >> 4), idesc,
                                           tsfa + uint32_t(4 * j), tsfb + uint32_t(4 * copies * j), (i | j) != 0);
                    } else if constexpr (KIND == 0) {
                        // descriptors advance by 32 bytes per block within a 128-k chunk
                        // (2 in their 16-byte address field) and by a chunk after four
#pragma unroll
                        for (int kb = 0; kb < kBsStageBlocks; ++kb)
                            if (kb < nb)
                                umma_bs<0>(d_t, ad0 + uint64_t(((kb >> 2) * kBsAChunk + (kb & 3) * 32) >> 4),
                                           bd0 + uint64_t(((kb >> 2) * (N * 128) + (kb & 3) * 32) >> 4),
                                           idesc | bs_sfid(uint32_t(kb & 3)), tsfa + uint32_t(4 * (kb >> 2)),
                                           tsfb + uint32_t(4 * copies * (kb >> 2)), (i | kb) != 0);
                    } else {
                        // four MMAs of 64 k (blocks 2j, 2j + 1: factor bytes 2 (j & 1), +1)
#pragma unroll
                        for (int j = 0; j < kBsStageBlocks / 2; ++j)
                            if (2 * j < nb)
                                umma_bs<1>(d_t, ad0 + uint64_t((j * 32) >> 4), bd0 + uint64_t((j * 32) >> 4),
                                           idesc | bs_sfid(uint32_t(2 * (j & 1))), tsfa + uint32_t(4 * (j >> 1)),
                                           tsfb + uint32_t(4 * copies * (j >> 1)), (i | j) != 0);
                    }
                    tc_commit(empty_b(c));
                    if (++c == R) {
                        c = 0;
                        ph ^= 1u;
                    }
                }
                if (ok) tc_commit(dready_b(db));
            }
            // every issued MMA has completed before the allocation is released
            tc_commit(fin_b);
        }
        __syncwarp();
        mbar_wait_sleep(fin_b, 0, S.status);
    } else if (warp < kBsFirstEpi) {
        // ------------------------------------------------ scale-factor warps
        // Per stage, once its bytes have landed: this quadrant's weight rows'
        // scales (from the TMA box) and X's factor cells (from the prepared X)
        // into the slot's factor columns, for every lane of the quadrant.
        const int q = warp & 3;
        const int r = 32 * q + lane;
        const uint32_t lane_addr = uint32_t(32 * q) << 16;
        const uint32_t sf0c = tbase + lane_addr + uint32_t(bs_sf0(KIND, npad));
        BsCursor<G> cur;
        cur.start(S);
        int it = 0, tc = 0, c = 0;
        uint32_t ph = 0;
        bool nan = false;
        for (; cur.valid(S); cur.next(S), ++it) {
            // the slot's previous stage was consumed before its bytes were requested again
            if (!wait(full_b(c), ph)) break;
            uint8_t* slot = smem + c * slot_bytes;
            const uint32_t tsfa = sf0c + sfcols * uint32_t(c);
            const uint32_t tsfb = tsfa + uint32_t(4 * bs_groups(KIND));
            if constexpr (KIND == 2) {
                // the stage's 16 E4M3 scales of row r: NaN flags the row; a
                // negative scale is folded into its 16 codes (sign bits flipped
                // in the slot's A tile, 128-byte swizzled) and used as |scale|
                const uint4 f = *reinterpret_cast<const uint4*>(slot + abytes + bbytes + 16 * r);
                const uint32_t w[4] = {f.x, f.y, f.z, f.w};
                uint32_t neg = 0u;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t mag = w[j] & 0x7F7F7F7Fu;
                    nan |= __vcmpeq4(mag, 0x7F7F7F7Fu) != 0u;
                    neg |= w[j] & 0x80808080u;
                    tmem_st4(tsfa + uint32_t(4 * j), mag, mag, mag, mag);
                }
                bool flipped = false;
                if (neg) {
                    // rare: fold each negative scale into its block's codes
#pragma unroll 1
                    for (int blk = 0; blk < 16; ++blk) {
                        const uint32_t b = (w[blk >> 2] >> (8 * (blk & 3))) & 0xFFu;
                        if ((b & 0x80u) && (b & 0x7Fu) != 0x7Fu) {
                            uint64_t* codes = reinterpret_cast<uint64_t*>(
                                slot + r * 128 + ((((blk >> 1) ^ (r & 7))) << 4) + 8 * (blk & 1));
                            *codes ^= 0x8888888888888888ull;
                            flipped = true;
                        }
                    }
                }
                if (flipped) fence_proxy_async_smem();
            } else {
                const uint2 f = *reinterpret_cast<const uint2*>(slot + abytes + bbytes + 16 * r + (cur.kb() & 8));
                nan |= has_byte_ff(f.x) || has_byte_ff(f.y);
                tmem_st4(tsfa, f.x, f.x, f.x, f.x);
                tmem_st4(tsfa + 4u, f.y, f.y, f.y, f.y);
            }
            const uint8_t* cells = slot + abytes + brows + 16 * lane;
#pragma unroll
            for (int gh = 0; gh < 8; ++gh)
                if (gh < bs_groups(KIND) * copies) {
                    const uint4 v = *reinterpret_cast<const uint4*>(cells + kBsCopyBytes * gh);
                    tmem_st4(tsfb + uint32_t(4 * gh), v.x, v.y, v.z, v.w);
                }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(sfok_b(c));
            if (++c == R) {
                c = 0;
                ph ^= 1u;
            }
            if (cur.i == cur.R.nst - 1) {
                // the tile's NaN-scale flags, once the epilogue is done with the slot's previous tile
                const int db = tc & 1;
                if (tc >= 2 && !wait(dfree_b(db), ((tc >> 1) - 1) & 1)) break;
                nanflags[db * kBsRows + r] = nan ? 1 : 0;
                __syncwarp();
                if (lane == 0) mbar_arrive(flags_b(db));
                nan = false;
                ++tc;
            }
        }
    } else {
        // ------------------------------------------------------- epilogue
        const int q = warp & 3;
        const int r = 32 * q + lane;
        const uint32_t lane_addr = uint32_t(32 * q) << 16;
        bool waited_pdl = false;
        int tc = 0;
        int ychunk = 0;  // output chunks staged so far (buffer parity)
        for (int w = int(blockIdx.x); w < S.items; w += int(gridDim.x), ++tc) {
            const Problem& pb = S.p[find_problem(S, w)];
            const int wl = w - pb.item_begin;
            const BsItem RI = bs_item(pb, wl);
            const int64_t n0 = int64_t(RI.tile) * kBsRows;
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
            const int64_t Ny = pb.N;
            const int nsplit = pb.nsplit;
            const float gs = pb.gscale;
            float* const ycol = pb.y + n0 + r;  // this lane's column of Y
            float* mine = pb.part + int64_t(wl) * M * kBsRows;
            const uint32_t dcol = tbase + lane_addr + (db ? d1col : 0u);
            // Y rows c0 .. c0 + 15 from their accumulators: the 16 rows' unscale
            // factors are loaded together first (read-only here: written by the
            // preparation kernel), so that no store waits on a load behind it
            auto put16 = [&](int c0, const float (&acc)[16]) {
                float xs[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) xs[c] = c0 + c < M ? __ldg(xun + c0 + c) : 0.f;
                if (kYB && S.y_tma && nsplit == 1) {
                    // single GEMM, no split: the 16 x 32 box of this warp through
                    // shared memory and one tensor store (rows of Y lie N floats
                    // apart: one thread store per row and lane group stalls on each)
                    if (lane == 0) bulk_wait_read_1();  // the buffer's store two chunks ago has read it
                    __syncwarp();
                    float* buf = ystage + (q * 2 + (ychunk & 1)) * (16 * 32);
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const float v = nan ? __int_as_float(0x7FC00000) : acc[c];
                        buf[c * 32 + lane] = KIND == 2 ? (v * xs[c]) * gs : v * xs[c];
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        // boxes reaching past N or M are clipped by the copy; one
                        // group per chunk, so that the waits above count chunks
                        if (n0 + 32 * q < Ny && c0 < M) tma_store_2d(&S.tm_y, smem_u32(buf), int(n0 + 32 * q) * 4, c0);
                        bulk_commit();
                    }
                    ++ychunk;
                    return;
                }
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const int m = c0 + c;
                    if (m < M) {
                        const float v = nan ? __int_as_float(0x7FC00000) : acc[c];
                        if (nsplit == 1) {
                            if (r < rows) ycol[int64_t(m) * Ny] = KIND == 2 ? (v * xs[c]) * gs : v * xs[c];
                        } else {
                            __stcg(mine + int64_t(m) * kBsRows + r, v);
                        }
                    }
                }
            };
            if constexpr (KIND == 3) {
                // one term: the next 16 columns' tensor-memory load is in flight
                // while this chunk is stored
                uint32_t d[16];
                tmem_ld16(dcol, d);
#pragma unroll 1
                for (int c0 = 0; c0 < npad; c0 += 16) {
                    tmem_wait_ld_into(d);
                    float acc[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) acc[c] = __uint_as_float(d[c]);
                    if (c0 + 16 < npad) tmem_ld16(dcol + uint32_t(c0 + 16), d);
                    put16(c0, acc);
                }
            } else {
#pragma unroll 1
                for (int c0 = 0; c0 < npad; c0 += 16) {
                    // the sum of the rows' T term columns, in term order
                    float acc[16];
#pragma unroll 1
                    for (int t = 0; t < T; ++t) {
                        uint32_t d[16];
                        tmem_ld16(dcol + uint32_t(t * npad + c0), d);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 16; ++c)
                            acc[c] = t == 0 ? __uint_as_float(d[c]) : acc[c] + __uint_as_float(d[c]);
                    }
                    put16(c0, acc);
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
                if (lane == 0) last = atomicAdd(pb.counters + 4 * RI.tile + q, 1) == pb.nsplit - 1;
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
                    __threadfence();
                    if (r < rows) {
                        // 8 rows at a time, so that their loads are in flight
                        // together; each row summed in split order
                        const float* pt = pb.part + int64_t(RI.tile) * M * kBsRows + r;
                        const int64_t sstride = int64_t(pb.ntiles) * M * kBsRows;
#pragma unroll 1
                        for (int m0 = 0; m0 < M; m0 += 8) {
                            float s[8];
#pragma unroll
                            for (int j = 0; j < 8; ++j) s[j] = 0.f;
#pragma unroll 4
                            for (int sp = 0; sp < nsplit; ++sp) {
                                float v[8];
#pragma unroll
                                for (int j = 0; j < 8; ++j)
                                    v[j] = m0 + j < M ? __ldcg(pt + sp * sstride + int64_t(m0 + j) * kBsRows) : 0.f;
#pragma unroll
                                for (int j = 0; j < 8; ++j) s[j] += v[j];
                            }
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const int m = m0 + j;
                                if (m < M) {
                                    const float xm = __ldg(xun + m);
                                    ycol[int64_t(m) * Ny] = KIND == 2 ? (s[j] * xm) * gs : s[j] * xm;
                                }
                            }
                        }
                    }
                    if (lane == 0) pb.counters[4 * RI.tile + q] = 0;  // ready for the next call
                }
            }
        }
        if (kYB && S.y_tma && lane == 0) bulk_wait_all();  // the staged stores have landed
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tbase, kBsTmemCols);
}
