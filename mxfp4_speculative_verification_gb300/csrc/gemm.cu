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
//  * that kernel takes passes of at most 8 rows; passes of 9..64 rows run on
//    the block-scaled tcgen05 kernel of gemm_bs.cuh (E2M1 weights and their
//    E8M0 scales straight into the tensor core, X as a sum of narrow terms;
//    `bs_kind_for`), fed by the same preparation kernel in its own layout.
//    The earlier tcgen05 kernel of gemm_umma.cuh (weights decoded to fp16 in
//    tensor memory) stays available behind MXS_GEMM_PATH=umma.
//
// Files: gemm_common.cuh (problem table, TMA helpers, work items),
// gemm_mma.cuh (the mma.sync kernel), gemm_bs.cuh (the block-scaled kernel),
// gemm_umma.cuh (the fp16 tcgen05 kernel), gemm_prep.cuh (X preparation);
// this file holds the host launchers.
#include <cuda.h>  // CUtensorMap and the tensor-map enums (types only)

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include <cuda_fp16.h>

#include "mxs_device.cuh"
#include "mxs_internal.h"

namespace mxs {

constexpr int kMaxDevices = 64;
constexpr int kMaxSplit = 32;
constexpr int64_t kMaxSplitItems = 2048;         // bound on tiles x splits when K is split
constexpr int64_t kBsMaxSplitItems = 304;        // the same for the block-scaled kernel (2 per SM)

#include "gemm_common.cuh"
#include "gemm_mma.cuh"
#include "gemm_umma.cuh"
#include "gemm_bs.cuh"
#include "gemm_prep.cuh"

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

// Largest split-K work-item count of the block-scaled kernel (0 if it never splits).
static int64_t bs_split_items_cap(int64_t N, int64_t K) {
    const int64_t ntiles = (N + kBsRows - 1) / kBsRows;
    const int64_t stages = (K / 32 + kBsStageBlocks - 1) / kBsStageBlocks;
    const int64_t ns = std::min<int64_t>(
        {int64_t(kMaxSplit), stages, std::max<int64_t>(1, kBsMaxSplitItems / ntiles)});
    return ns > 1 ? ntiles * ns : 0;
}

static int bs_kind_for(int64_t rows_left, int64_t K, const void* nib);
static bool bs_nv_for(int64_t rows_left, int64_t K, const void* nib);

// Whether a call of M rows may run a block-scaled pass (sizes its workspace;
// the nibbles' alignment is not known yet, so assume the best).
static bool bs_may_run(int64_t M, int64_t K) { return bs_kind_for(M, K, nullptr) >= 0; }
static bool bs_nv_may_run(int64_t M, int64_t K) { return bs_nv_for(M, K, nullptr); }

// Bytes of X prepared for the block-scaled kernel (passes of at most mc
// rows, either kind).
static size_t bs_x_bytes(int64_t mc, int64_t K, bool nv = false) {
    const int m = int(std::min<int64_t>(mc, kBsMaxNpad));
    const int per_stage = nv ? bs_bstage_bytes(2, bs_npad(2, std::min(m, bs_max_rows(2))))
                             : std::max(bs_bstage_bytes(0, bs_npad(0, m)),
                                        bs_bstage_bytes(1, bs_npad(1, std::min(m, kBsF4MaxRows))));
    return size_t((K + 255) / 256) * size_t(per_stage);
}

GemmWorkspace gemm_workspace_layout(int64_t M, int64_t N, int64_t K, bool scales_aligned, int sdiv) {
    GemmWorkspace w{};
    const bool nv = sdiv == 16;  // NVFP4: scale bytes per 16 k
    const int64_t nblk = K / sdiv;
    const int64_t mc = std::min<int64_t>(M, kGemmMaxRowsPerPass);
    const int64_t mcb = std::min<int64_t>(M, kBsMaxNpad);
    w.repack_scales = !(K % (16 * sdiv) == 0 && scales_aligned);
    w.sc_pitch = w.repack_scales ? int(align_up(size_t(nblk), 16)) : int(nblk);
    size_t off = 0;
    w.xf_off = off;
    off = align_up(off + std::max(size_t(kGemmMaxRowsPerPass) * align_up(size_t(K), 512) * 2,
                                  (nv ? bs_nv_may_run(M, K) : bs_may_run(M, K)) ? bs_x_bytes(mcb, K, nv) : size_t(0)),
                   256);
    w.xun_off = off;
    off = align_up(off + kBsMaxNpad * sizeof(float), 256);
    // counters and partial tiles, sized for any tile height a pass may use
    // (the block-scaled kernel counts each 32-row quarter of a tile apart)
    int64_t ncnt = 0, part = 0;
    for (int bn : {64, 128}) {
        const int64_t cap = split_items_cap(N, K, bn);
        if (cap > 0) {
            ncnt = std::max<int64_t>(ncnt, (N + bn - 1) / bn);
            part = std::max<int64_t>(part, cap * mc * bn);
        }
    }
    if (nv ? bs_nv_may_run(M, K) : bs_may_run(M, K)) {
        const int64_t cap = bs_split_items_cap(N, K);
        if (cap > 0) {
            ncnt = std::max<int64_t>(ncnt, 4 * ((N + kBsRows - 1) / kBsRows));
            part = std::max<int64_t>(part, cap * mcb * kBsRows);
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

// 3-D tensor map over packed E2M1 nibbles [rows, K] for the block-scaled
// kernel: dims (128 codes, rows, K / 128 chunks), each request of the
// 16U4_ALIGN16B type spreading 16 codes (8 bytes) over 16 bytes of shared
// memory; boxes of 128 codes x 128 rows x `chunks`, 128-byte swizzle.  Needs
// K % 128 == 0 and a 32-byte aligned base (the type's rules).
static bool make_map_e2m1_spread(CUtensorMap* map, const void* base, int64_t rows, int64_t K, uint32_t chunks) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    cuuint64_t dims[3] = {128, cuuint64_t(rows), cuuint64_t(K / 128)};
    cuuint64_t strides[2] = {cuuint64_t(K / 2), 64};
    cuuint32_t box[3] = {128, uint32_t(kBsRows), chunks};
    cuuint32_t estr[3] = {1, 1, 1};
    std::memset(map, 0, sizeof(*map));
    return f(map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Per-device launch facts of one kernel instantiation, computed on first use.
struct LaunchFacts {
    std::atomic<int> sms[kMaxDevices];
    std::atomic<int> occ[kMaxDevices];
};

// Split of K: the count whose busiest CTA streams the fewest stages, with a
// small charge per extra work item for its partial-tile round trip.
static void choose_split(int64_t ntiles, int stages_total, int64_t grid_cap, int64_t items_cap,
                         int& nsplit, int& per_split, double item_cost = 0.35) {
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
        const double cost = per_cta * (sps + (ns > 1 ? item_cost : 0.0));
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
    int sdiv = 32;       // k per scale byte: 32 (MXFP4, E8M0) or 16 (NVFP4, E4M3)
    float gscale = 1.f;  // NVFP4 tensor scale
};

// Fill the launch's problem table for tiles of BN rows.
// bs: the block-scaled kernel (256-k stages, scales read in place), 1 for
// its mxf8f6f4 kind (padded E2M1 boxes), 2, 3 and 4 for its mxf4, mxf4nvf4
// and W4A4 kinds (packed boxes).
template <int G>
static cudaError_t build_problems(ProblemSet<G>& S, const HostGemm* gs, int count, int M,
                                  int32_t* status, int BN, int64_t resident, int* sched,
                                  int bs = 0) {
    std::memset(&S, 0, sizeof(S));
    S.count = count;
    S.M = M;
    S.status = status;
    S.sched = sched;
    // bounded waits: the limit, and (tests only) a stage CTA 0 leaves out
    const long long wl = std::atoll(std::getenv("MXS_GEMM_WAIT_LIMIT_NS") ? std::getenv("MXS_GEMM_WAIT_LIMIT_NS") : "0");
    S.wait_ns = wl > 0 ? (unsigned long long)wl : kWaitLimitNs;
    S.skip_stage = env_int("MXS_GEMM_TEST_SKIP_STAGE", -1);
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
        p.gscale = h.gscale;
        const int sblk = bs ? kBsStageBlocks : kStageBlocks;
        const int stages_total = (p.nblk + sblk - 1) / sblk;
        p.nsplit = 1;
        p.stages_per_split = stages_total;
        if (h.items_cap > 0) {
            choose_split(p.ntiles, stages_total, resident, h.items_cap, p.nsplit, p.stages_per_split,
                         bs ? 0.7 : 0.35);
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
        if (bs) {
            // weights: both 128-k chunks of a stage per request (padded E2M1 for
            // mxf8f6f4), or the packed bytes of the stage (mxf4); scales: 16
            // blocks x 128 rows per request (the rows are 16-byte aligned:
            // K % 512 == 0 in place, else realigned in the workspace)
            const bool wmap = bs == 1 ? make_map_e2m1_spread(&p.tm_w, h.nib, h.N, h.K, 2)
                                      : make_map(&p.tm_w, h.nib, h.N, h.K / 2, h.K / 2, kBoxBytes, uint32_t(kBsRows), true);
            if (!wmap || !make_map(&p.tm_s, h.sc, h.N, h.K / h.sdiv, h.sc_pitch, 16, uint32_t(kBsRows), false))
                return cudaErrorInvalidValue;
            continue;
        }
        if (!make_map(&p.tm_w, h.nib, h.N, h.K / 2, h.K / 2, kBoxBytes, uint32_t(BN), true))
            return cudaErrorInvalidValue;
        // one 16-byte (MXFP4) or 32-byte (NVFP4) column of scales per 512-k stage
        if (!make_map(&p.tm_s, h.sc, h.N, h.K / h.sdiv, h.sc_pitch, h.sdiv == 16 ? 32 : 16, uint32_t(BN), false))
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

template <int NT, int RG, int KW, int STAGES, int G, bool NV = false>
static cudaError_t launch_main(const HostGemm* gs, int count, int M, int32_t* status,
                               int* sched, cudaStream_t stream) {
    using C = GemmCfg<NT, RG, KW, STAGES, NV>;
    auto kern = mxfp4_gemm_kernel<NT, RG, KW, STAGES, G, NV>;
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
template <int G, bool NV = false>
static cudaError_t launch_main_nt(int NT, const HostGemm* gs, int count, int M, int32_t* status,
                                  int* sched, cudaStream_t stream) {
    switch (NT) {
        case 1: return launch_main<1, 4, 2, 4, G, NV>(gs, count, M, status, sched, stream);
        case 2: return launch_main<2, 4, 2, 3, G, NV>(gs, count, M, status, sched, stream);
        case 3: return launch_main<3, 8, 2, 3, G, NV>(gs, count, M, status, sched, stream);
        case 4: return launch_main<4, 8, 2, 2, G, NV>(gs, count, M, status, sched, stream);
        default: return launch_main<8, 4, 2, 2, G, NV>(gs, count, M, status, sched, stream);
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

// Stage slots of the block-scaled kernel for a pass of npad rows;
// MXS_GEMM_BS_RINGS=c overrides it when c slots fit shared and tensor memory.
static int bs_ring_for(int kind, int npad, int ybytes) {
    const int c = env_int("MXS_GEMM_BS_RINGS", 0);
    if (c >= 2 && c <= kBsMaxRing && bs_smem_bytes(kind, npad, c, ybytes) <= kBsSmemAttr &&
        bs_tmem_need(kind, npad, c) <= int(kBsTmemCols))
        return c;
    return bs_ring(kind, npad, ybytes);
}

// Block-scaled kernel: one CTA per SM, 128-row tiles, K split only for a
// single GEMM whose tiles leave SMs idle.
template <int G, int KIND>
static cudaError_t launch_bs(const HostGemm* gs, int count, int M, int32_t* status, cudaStream_t stream) {
    auto kern = mxfp4_gemm_bs_kernel<G, KIND>;
    static LaunchFacts facts;
    int sms = 0, occ = 0;
    cudaError_t err = launch_facts(facts, kern, kBsThreads, kBsSmemAttr, sms, occ);
    if (err != cudaSuccess) return err;
    static thread_local ProblemSet<G>* S_buf = nullptr;
    if (!S_buf) S_buf = new ProblemSet<G>;
    err = build_problems(*S_buf, gs, count, M, status, kBsRows, int64_t(sms), nullptr, KIND == 0 ? 1 : KIND + 1);
    if (err != cudaSuccess) return err;
    const int npad = bs_npad(KIND, M);
    // single-GEMM launches keep room for the output staging where it costs
    // no stage slot, or where passes have 64 rows or more (their thread
    // stores of Y cost more than the slot); then, without a K split and with
    // 16-byte aligned rows of Y, Y goes out by tensor stores
    const int ybytes =
        G == 1 && (npad >= 64 || bs_ring(KIND, npad, kBsYStageBytes) == bs_ring(KIND, npad, 0)) ? kBsYStageBytes : 0;
    S_buf->y_tma = 0;
    if constexpr (G == 1) {
        const HostGemm& h = gs[0];
        if (ybytes && count == 1 && S_buf->p[0].nsplit == 1 && h.N % 4 == 0 &&
            (reinterpret_cast<uintptr_t>(h.y) & 15) == 0 && make_map(&S_buf->tm_y, h.y, M, h.N * 4, h.N * 4, 128, 16, false))
            S_buf->y_tma = 1;
    }
    S_buf->ring = bs_ring_for(KIND, npad, ybytes);
    const int64_t grid = std::min<int64_t>(S_buf->items, int64_t(sms));
    return launch_persistent(kern, *S_buf, kBsThreads, bs_smem_bytes(KIND, npad, S_buf->ring, ybytes), grid, stream);
}

template <int G>
static cudaError_t launch_bs_kind(int kind, const HostGemm* gs, int count, int M, int32_t* status,
                                  cudaStream_t stream) {
    if constexpr (G == 1) {
        if (kind == 2) return launch_bs<1, 2>(gs, count, M, status, stream);  // NVFP4: single calls only
    }
    if (kind == 3) return launch_bs<G, 3>(gs, count, M, status, stream);  // W4A4
    return kind ? launch_bs<G, 1>(gs, count, M, status, stream) : launch_bs<G, 0>(gs, count, M, status, stream);
}

// Every pass size the block-scaled kernel takes fits its shared and tensor memory.
static constexpr bool bs_shapes_fit() {
    for (int kind = 0; kind < 4; ++kind)
        for (int m = 1; m <= bs_max_rows(kind); ++m) {
            const int npad = bs_npad(kind, m);
            for (int yb = 0; yb <= kBsYStageBytes; yb += kBsYStageBytes) {
                const int rc = bs_ring(kind, npad, yb);
                if (bs_smem_bytes(kind, npad, rc, yb) > kBsSmemAttr || bs_tmem_need(kind, npad, rc) > int(kBsTmemCols) ||
                    rc > kBsMaxRing || rc < 3 || bs_slot_bytes(kind, npad) % 1024 != 0)
                    return false;
            }
        }
    return true;
}
static_assert(bs_shapes_fit(), "block-scaled kernel: a pass size exceeds shared or tensor memory");

// The kind of block-scaled pass that takes the next rows (rows_left of
// them), or -1 for the mma.sync / tcgen05 f16 kernels.  Passes of at least
// MXS_GEMM_BS_MIN rows (default 9) go to the block-scaled kernel: up to 32
// rows the mxf4 kind (any K, 16-byte aligned nibbles), beyond that
// mxf8f6f4, which needs K % 128 == 0 and 32-byte aligned nibbles (the padded
// TMA type's rules) and otherwise leaves the pass to the older kernels.
// MXS_GEMM_PATH=bs8 or bs4 forces one kind for every pass it can take
// (bs4: 32 rows at most per pass), bs the default choice at any row count,
// mma or umma the older kernels.
static int bs_kind_for(int64_t rows_left, int64_t K, const void* nib) {
    const bool f8_ok = K % 128 == 0 && (reinterpret_cast<uintptr_t>(nib) & 31) == 0;
    const bool f4_ok = K % 32 == 0 && (reinterpret_cast<uintptr_t>(nib) & 15) == 0;
    const char* path = std::getenv("MXS_GEMM_PATH");
    if (path && std::strcmp(path, "bs8") == 0) return f8_ok ? 0 : -1;
    if (path && std::strcmp(path, "bs4") == 0) return f4_ok ? 1 : -1;
    if (path && (std::strcmp(path, "mma") == 0 || std::strcmp(path, "umma") == 0)) return -1;
    const bool forced = path && std::strcmp(path, "bs") == 0;
    if (!forced && rows_left < env_int("MXS_GEMM_BS_MIN", 9)) return -1;
    if (rows_left <= kBsF4MaxRows) return f4_ok ? 1 : (f8_ok ? 0 : -1);
    return f8_ok ? 0 : -1;
}
// Rows of a block-scaled pass of the given kind.
static int64_t bs_pass_rows(int kind, int64_t rows_left) {
    if (kind == 3) {
        // W4A4: as few passes as 256 rows allow, of equal size (rounded up to
        // 16): 320 rows as 2 x 160 keep two D buffers in tensor memory, where
        // 256 + 64 would run the first pass on one
        const int64_t passes = (rows_left + kBsW4MaxRows - 1) / kBsW4MaxRows;
        return std::min<int64_t>(rows_left, ((rows_left + passes - 1) / passes + 15) / 16 * 16);
    }
    return std::min<int64_t>(bs_max_rows(kind), rows_left);
}

// Whether the next NVFP4 pass (rows_left rows) takes the block-scaled kernel
// (kind::mxf4nvf4, passes of at most 64 rows): 16-byte aligned nibbles, and
// passes of at least MXS_GEMM_NV_BS_MIN rows (default 1); MXS_GEMM_PATH=mma
// keeps every pass on the mma.sync kernel, =bs sends every pass it can.
static bool bs_nv_for(int64_t rows_left, int64_t K, const void* nib) {
    const bool ok = K % 32 == 0 && (reinterpret_cast<uintptr_t>(nib) & 15) == 0;
    const char* path = std::getenv("MXS_GEMM_PATH");
    if (path && std::strcmp(path, "mma") == 0) return false;
    if (path && (std::strcmp(path, "bs") == 0 || std::strcmp(path, "bs4") == 0)) return ok;
    return ok && rows_left >= env_int("MXS_GEMM_NV_BS_MIN", 1);
}

// For a pass the block-scaled kernel does not take: whether the fp16
// tcgen05 kernel runs it instead of mma.sync (more than 24 rows, where the
// m16n8k16 issue rate rather than HBM bounds mma.sync).  MXS_GEMM_PATH=mma|umma
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
    const int rows = Q.bs_npad > 0 ? Q.bs_npad : (Q.umma_npad > 0 ? Q.umma_npad : 8 * Q.NT);
    cfg.gridDim = dim3(unsigned(Q.njobs * rows + 1 + Q.repack_ctas), 1, 1);
    // block-scaled passes: 256 threads, so that a preparation CTA and a CTA of
    // the main kernel (launched early through PDL) fit one SM together
    cfg.blockDim = dim3(Q.bs_npad > 0 ? kPrepThreadsBs : kPrepThreads, 1, 1);
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
    bool scales_realigned = false;
    for (int64_t m0 = 0, mc = 0; m0 < M; m0 += mc) {
        const int kind = bs_kind_for(M - m0, K, nibbles);
        // the scales are realigned once, by the first pass that reads them;
        // every pass that streams the realigned copy waits for the preparation
        // kernel before its first scale request (its completion implies that
        // of every earlier kernel of the call)
        const bool repack = ws.repack_scales && !scales_realigned;
        scales_realigned = true;
        if (kind >= 0) {
            // block-scaled pass: its own X layout
            mc = bs_pass_rows(kind, M - m0);
            PrepSet Q{};
            Q.job[0].x = x + m0 * K;
            Q.job[0].xf = xf;
            Q.job[0].xun = xun;
            Q.job[0].K = int(K);
            Q.njobs = 1;
            Q.M = int(mc);
            Q.NT = 1;
            Q.bs_npad = bs_npad(kind, int(mc));
            Q.bs_kind = kind;
            Q.counters = counters;
            Q.ncounters = ws.n_counters;
            if (repack) {
                Q.sc_in = scales;
                Q.N = N;
                Q.nblk = nblk;
                Q.sc_pitch = ws.sc_pitch;
                Q.sc_out = sc_aligned;
                Q.repack_ctas = int(std::min<int64_t>((N * ws.sc_pitch + kPrepThreadsBs - 1) / kPrepThreadsBs, 1024));
            }
            cudaError_t err = launch_prep(Q, stream);
            if (err != cudaSuccess) return err;
            HostGemm h{};
            h.nib = nibbles;
            h.sc = ws.repack_scales ? sc_aligned : scales;
            h.sc_pitch = ws.repack_scales ? ws.sc_pitch : nblk;
            h.sc_from_prep = ws.repack_scales;
            h.xf = xf;
            h.xun = xun;
            h.y = y + m0 * N;
            h.part = part;
            h.counters = counters;
            h.N = N;
            h.K = K;
            const int64_t cap = bs_split_items_cap(N, K);
            h.items_cap = (cap > 0 && ws.n_counters >= 4 * ((N + kBsRows - 1) / kBsRows)) ? cap : 0;
            err = launch_bs_kind<1>(kind, &h, 1, int(mc), dev_status, stream);
            if (err != cudaSuccess) return err;
            continue;
        }
        mc = std::min<int64_t>(kGemmMaxRowsPerPass, M - m0);
        const int NT = tiles_nt(int(mc));
        const int bn = bn_for_nt(NT);
        // the workspace holds partial tiles for mc0 rows and tile height bn
        int64_t items_cap = split_items_cap(N, K, bn);
        if (ws.n_counters < (N + bn - 1) / bn || mc > mc0) items_cap = 0;
        const bool umma = use_umma(int(mc), (N + kUBN - 1) / kUBN, false);
        PrepSet Q{};
        Q.job[0].x = x + m0 * K;
        Q.job[0].xf = xf;
        Q.job[0].xun = xun;
        Q.job[0].K = int(K);
        Q.njobs = 1;
        Q.M = int(mc);
        Q.NT = NT;
        Q.umma_npad = umma ? umma_npad(int(mc)) : 0;
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
        h.sc_from_prep = ws.repack_scales;
        h.xf = xf;
        h.xun = xun;
        h.y = y + m0 * N;
        h.part = part;
        h.counters = counters;
        h.N = N;
        h.K = K;
        h.items_cap = items_cap;
        err = umma ? launch_umma_np<1>(umma_npad(int(mc)), &h, 1, int(mc), dev_status, stream)
                   : launch_main_nt<1>(NT, &h, 1, int(mc), dev_status, nullptr, stream);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

// NVFP4 weights ("Module 11 ...", §12: E2M1 in blocks of 16 sharing an E4M3
// scale, one FP32 scale per tensor): passes of up to 64 rows on the mma.sync
// kernel, each block's scale folded into the decoded fp16 weights.
cudaError_t gemm_run_nv(const uint16_t* x, const uint8_t* nibbles, const uint8_t* scales, float global_scale,
                        float* y, int64_t M, int64_t N, int64_t K, void* workspace, const GemmWorkspace& ws,
                        int32_t* dev_status, cudaStream_t stream) {
    uint8_t* wsb = static_cast<uint8_t*>(workspace);
    uint16_t* xf = reinterpret_cast<uint16_t*>(wsb + ws.xf_off);
    float* xun = reinterpret_cast<float*>(wsb + ws.xun_off);
    int* counters = reinterpret_cast<int*>(wsb + ws.cnt_off);
    float* part = reinterpret_cast<float*>(wsb + ws.part_off);
    uint8_t* sc_aligned = ws.repack_scales ? wsb + ws.sc_off : nullptr;
    const int nsb = int(K / 16);  // scale bytes per row
    const int64_t mc0 = std::min<int64_t>(M, kGemmMaxRowsPerPass);
    bool scales_realigned = false;
    for (int64_t m0 = 0, mc = 0; m0 < M; m0 += mc) {
        if (bs_nv_for(M - m0, K, nibbles)) {
            // block-scaled pass (kind::mxf4nvf4): its own X layout
            mc = bs_pass_rows(2, M - m0);
            const bool repack = ws.repack_scales && !scales_realigned;
            scales_realigned = true;
            PrepSet Q{};
            Q.job[0].x = x + m0 * K;
            Q.job[0].xf = xf;
            Q.job[0].xun = xun;
            Q.job[0].K = int(K);
            Q.njobs = 1;
            Q.M = int(mc);
            Q.NT = 1;
            Q.bs_npad = bs_npad(2, int(mc));
            Q.bs_kind = 2;
            Q.counters = counters;
            Q.ncounters = ws.n_counters;
            if (repack) {
                Q.sc_in = scales;
                Q.N = N;
                Q.nblk = nsb;
                Q.sc_pitch = ws.sc_pitch;
                Q.sc_out = sc_aligned;
                Q.repack_ctas = int(std::min<int64_t>((N * ws.sc_pitch + kPrepThreadsBs - 1) / kPrepThreadsBs, 1024));
            }
            cudaError_t err = launch_prep(Q, stream);
            if (err != cudaSuccess) return err;
            HostGemm h{};
            h.nib = nibbles;
            h.sc = ws.repack_scales ? sc_aligned : scales;
            h.sc_pitch = ws.sc_pitch;
            h.sc_from_prep = ws.repack_scales;
            h.xf = xf;
            h.xun = xun;
            h.y = y + m0 * N;
            h.part = part;
            h.counters = counters;
            h.N = N;
            h.K = K;
            h.sdiv = 16;
            h.gscale = global_scale;
            const int64_t cap = bs_split_items_cap(N, K);
            h.items_cap = (cap > 0 && ws.n_counters >= 4 * ((N + kBsRows - 1) / kBsRows)) ? cap : 0;
            err = launch_bs_kind<1>(2, &h, 1, int(mc), dev_status, stream);
            if (err != cudaSuccess) return err;
            continue;
        }
        mc = std::min<int64_t>(kGemmMaxRowsPerPass, M - m0);
        const int NT = tiles_nt(int(mc));
        const int bn = bn_for_nt(NT);
        int64_t items_cap = split_items_cap(N, K, bn);
        if (ws.n_counters < (N + bn - 1) / bn || mc > mc0) items_cap = 0;
        const bool repack = ws.repack_scales && !scales_realigned;
        scales_realigned = true;
        PrepSet Q{};
        Q.job[0].x = x + m0 * K;
        Q.job[0].xf = xf;
        Q.job[0].xun = xun;
        Q.job[0].K = int(K);
        Q.njobs = 1;
        Q.M = int(mc);
        Q.NT = NT;
        Q.counters = counters;
        Q.ncounters = ws.n_counters;
        if (repack) {
            Q.sc_in = scales;
            Q.N = N;
            Q.nblk = nsb;
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
        h.sc_from_prep = ws.repack_scales;
        h.xf = xf;
        h.xun = xun;
        h.y = y + m0 * N;
        h.part = part;
        h.counters = counters;
        h.N = N;
        h.K = K;
        h.items_cap = items_cap;
        h.sdiv = 16;
        h.gscale = global_scale;
        err = launch_main_nt<1, true>(NT, &h, 1, int(mc), dev_status, nullptr, stream);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

// ------------------------------------------------------------------ grouped
// Independent GEMMs sharing M <= 64: each distinct X is converted once, then
// persistent launches of up to kGroupMax GEMMs stream every weight matrix
// through the same shared-memory ring.
constexpr int kGroupMax = 84;
static_assert(sizeof(ProblemSet<kGroupMax>) <= 32764, "the problem table is a kernel parameter (32764 bytes at most)");

// Bytes of one prepared X (any layout) for an X of M rows.
static size_t xf_bytes(int64_t M, int64_t K) {
    const int mc0 = int(std::min<int64_t>(M, kGemmMaxRowsPerPass));
    const int rows = std::max(8 * tiles_nt(mc0), umma_npad(mc0));
    return std::max(size_t(rows) * align_up(size_t(K), 512) * 2,
                    bs_may_run(M, K) ? bs_x_bytes(std::min<int64_t>(M, kBsMaxNpad), K) : size_t(0));
}

// X of one W4A4 pass (the quantised rows of up to 256 rows) and its row factors
static size_t xf_w4a4_bytes(int64_t M, int64_t K) {
    const int m = int(std::min<int64_t>(M, kBsW4MaxRows));
    return size_t((K + 255) / 256) * size_t(bs_bstage_bytes(3, bs_npad(3, m)));
}

size_t gemm_grouped_workspace(const GroupedGemm* gs, int count, int64_t M, bool w4a4) {
    size_t off = 0;
    for (int i = 0; i < count; ++i) {
        bool seen = false;
        for (int j = 0; j < i && !seen; ++j) seen = gs[j].x == gs[i].x && gs[j].K == gs[i].K;
        if (seen) continue;
        off = align_up(off + (w4a4 ? xf_w4a4_bytes(M, gs[i].K) : xf_bytes(M, gs[i].K)), 256);
        off = align_up(off + size_t(w4a4 ? kBsW4MaxRows : kBsMaxNpad) * sizeof(float), 256);
    }
    // one item claim counter per launch of a pass
    return align_up(off + size_t((count + kGroupMax - 1) / kGroupMax) * sizeof(int), 256);
}

cudaError_t gemm_grouped_run(const GroupedGemm* gs, int count, int64_t M, void* workspace,
                             int32_t* dev_status, cudaStream_t stream, bool w4a4) {
    uint8_t* wsb = static_cast<uint8_t*>(workspace);
    // distinct activations, in first-use order; X space sized for the largest pass
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
            off = align_up(off + (w4a4 ? xf_w4a4_bytes(M, gs[i].K) : xf_bytes(M, gs[i].K)), 256);
            J.xun = reinterpret_cast<float*>(wsb + off);
            off = align_up(off + size_t(w4a4 ? kBsW4MaxRows : kBsMaxNpad) * sizeof(float), 256);
            found = int(jobs.size());
            jobs.push_back(J);
        }
        xid[i] = found;
    }
    int* sched = reinterpret_cast<int*>(wsb + off);  // one claim counter per launch of a pass
    const int nlaunch = (count + kGroupMax - 1) / kGroupMax;
    std::vector<HostGemm> hs(count);
    // rows are processed up to 128 (block-scaled kernel) or 64 at a time; each
    // pass converts its rows of every distinct X, then streams every weight
    // matrix once
    for (int64_t m0 = 0, mcl = 0; m0 < M; m0 += mcl) {
        // one kind for every GEMM of the pass, or none if they would differ
        // (W4A4: the quantised-X kind for every pass)
        int kind = w4a4 ? 3 : (count > 0 ? bs_kind_for(M - m0, gs[0].K, gs[0].nibbles) : -1);
        for (int i = 1; i < count && kind >= 0 && !w4a4; ++i)
            if (bs_kind_for(M - m0, gs[i].K, gs[i].nibbles) != kind) kind = -1;
        const bool bs = kind >= 0;
        mcl = bs ? bs_pass_rows(kind, M - m0) : std::min<int64_t>(kGemmMaxRowsPerPass, M - m0);
        const int mc = int(mcl);
        const int NT = tiles_nt(mc);
        const bool umma = !bs && use_umma(mc, 0, true);
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
            Q.bs_npad = bs ? bs_npad(kind, mc) : 0;
            Q.bs_kind = bs ? kind : 0;
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
            int* claim = (umma || bs) ? nullptr : sched_or_null(sched + l);
            // claimed in table order: longest items (largest K) first
            if (claim)
                std::stable_sort(hs.begin() + b, hs.begin() + e,
                                 [](const HostGemm& u, const HostGemm& v) { return u.K > v.K; });
            cudaError_t err =
                bs     ? launch_bs_kind<kGroupMax>(kind, hs.data() + b, e - b, mc, dev_status, stream)
                : umma ? launch_umma_np<kGroupMax>(umma_npad(mc), hs.data() + b, e - b, mc, dev_status, stream)
                       : launch_main_nt<kGroupMax>(NT, hs.data() + b, e - b, mc, dev_status, claim, stream);
            if (err != cudaSuccess) return err;
        }
    }
    return cudaSuccess;
}

// ---------------------------------------------------------------------------
// W4A4 ("Module 11 ...", §12: MX-FP4 weights and activations): X quantised
// by the pack rule, block by block, then the block-scaled kind::mxf4 kernel
// with one term, so that N = the pass's rows and W is streamed once for up
// to 256 rows.  Its own workspace: the quantised X of a pass of up to 256
// rows, per-row factors, split-K counters and partial tiles, realigned scales.
// ---------------------------------------------------------------------------
GemmWorkspace gemm_w4a4_workspace_layout(int64_t M, int64_t N, int64_t K, bool scales_aligned) {
    GemmWorkspace w{};
    const int64_t nblk = K / 32;
    const int64_t mc = std::min<int64_t>(M, kBsW4MaxRows);
    const int npad = bs_npad(3, int(mc));
    w.repack_scales = !(K % 512 == 0 && scales_aligned);
    w.sc_pitch = w.repack_scales ? int(align_up(size_t(nblk), 16)) : int(nblk);
    size_t off = 0;
    w.xf_off = off;
    off = align_up(off + size_t((K + 255) / 256) * size_t(bs_bstage_bytes(3, npad)), 256);
    w.xun_off = off;
    off = align_up(off + size_t(kBsW4MaxRows) * sizeof(float), 256);
    const int64_t cap = bs_split_items_cap(N, K);
    w.cnt_off = off;
    w.n_counters = cap > 0 ? int(4 * ((N + kBsRows - 1) / kBsRows)) : 0;
    off = align_up(off + size_t(w.n_counters) * sizeof(int), 256);
    w.part_off = off;
    off = align_up(off + size_t(cap > 0 ? cap * mc * kBsRows : 0) * sizeof(float), 256);
    w.sc_off = off;
    if (w.repack_scales) off = align_up(off + size_t(N) * size_t(w.sc_pitch), 256);
    w.bytes = off;
    return w;
}

cudaError_t gemm_run_w4a4(const uint16_t* x, const uint8_t* nibbles, const uint8_t* scales, float* y, int64_t M,
                          int64_t N, int64_t K, void* workspace, const GemmWorkspace& ws, int32_t* dev_status,
                          cudaStream_t stream) {
    uint8_t* wsb = static_cast<uint8_t*>(workspace);
    uint16_t* xf = reinterpret_cast<uint16_t*>(wsb + ws.xf_off);
    float* xun = reinterpret_cast<float*>(wsb + ws.xun_off);
    int* counters = reinterpret_cast<int*>(wsb + ws.cnt_off);
    float* part = reinterpret_cast<float*>(wsb + ws.part_off);
    uint8_t* sc_aligned = ws.repack_scales ? wsb + ws.sc_off : nullptr;
    bool scales_realigned = false;
    for (int64_t m0 = 0, mc = 0; m0 < M; m0 += mc) {
        mc = bs_pass_rows(3, M - m0);
        const bool repack = ws.repack_scales && !scales_realigned;
        scales_realigned = true;
        PrepSet Q{};
        Q.job[0].x = x + m0 * K;
        Q.job[0].xf = xf;
        Q.job[0].xun = xun;
        Q.job[0].K = int(K);
        Q.njobs = 1;
        Q.M = int(mc);
        Q.NT = 1;
        Q.bs_npad = bs_npad(3, int(mc));
        Q.bs_kind = 3;
        Q.counters = counters;
        Q.ncounters = ws.n_counters;
        if (repack) {
            Q.sc_in = scales;
            Q.N = N;
            Q.nblk = int(K / 32);
            Q.sc_pitch = ws.sc_pitch;
            Q.sc_out = sc_aligned;
            Q.repack_ctas = int(std::min<int64_t>((N * ws.sc_pitch + kPrepThreadsBs - 1) / kPrepThreadsBs, 1024));
        }
        cudaError_t err = launch_prep(Q, stream);
        if (err != cudaSuccess) return err;
        HostGemm h{};
        h.nib = nibbles;
        h.sc = ws.repack_scales ? sc_aligned : scales;
        h.sc_pitch = ws.sc_pitch;
        h.sc_from_prep = ws.repack_scales;
        h.xf = xf;
        h.xun = xun;
        h.y = y + m0 * N;
        h.part = part;
        h.counters = counters;
        h.N = N;
        h.K = K;
        const int64_t cap = bs_split_items_cap(N, K);
        h.items_cap = (cap > 0 && ws.n_counters >= 4 * ((N + kBsRows - 1) / kBsRows)) ? cap : 0;
        err = launch_bs_kind<1>(3, &h, 1, int(mc), dev_status, stream);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

}  // namespace mxs
