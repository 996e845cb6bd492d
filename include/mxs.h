/*
 * mxs.h -- C ABI of the MXFP4 speculative-verification library (libmxs.so).
 *
 * The library runs the target model's verification step of speculative
 * decoding over OCP MX-FP4 weights on one GB300 (sm_103a):
 *
 *   mxfp4_pack         real weights -> E2M1 nibbles + E8M0 block scales
 *   mxfp4_verify_gemm  Y[M,N] = X[M,K] . dequant(W)^T, bf16 X, fp32 Y
 *                      (also grouped, without workspace, on NVFP4
 *                      weights: nvfp4_verify_gemm, and W4A4 with X
 *                      quantised to MX-FP4: mxfp4_verify_gemm_w4a4)
 *   spec_accept        left-to-right acceptance, residual / bonus sampling,
 *                      emission of 1..K+1 tokens per sequence (also from
 *                      logits under temperature / top-k / top-p:
 *                      spec_accept_logits, spec_sampling_law)
 *   mxfp4_kv_append,   the MX-FP4 KV cache of the verification block:
 *   spec_kv_commit,    append, keep what acceptance kept, read back
 *   mxfp4_kv_dequant
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *   allocates nothing and never synchronises: work is enqueued on `stream`
 *   (a cudaStream_t passed as void*; NULL = the legacy default stream) and
 *   the call returns after the launch.
 * - Host-side validation happens before any launch.  A non-zero mxs_status
 *   means nothing was enqueued.  MXS_ERR_CUDA reports a launch failure.
 * - Conditions only the device can see are OR-ed, stream-ordered, into
 *   `dev_status` (an int32 in device memory, nullable) as MXS_DEV_* bits.
 *   The library never clears it; the caller zeroes it when it wants a fresh
 *   reading.
 * - Layouts are row-major and dense (no strides).
 */
#ifndef MXS_H_
#define MXS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t mxs_status;

#define MXS_OK 0
#define MXS_ERR_INVALID_ARG 1   /* bad size, NULL pointer, K % 32 != 0, ... */
#define MXS_ERR_MISALIGNED 2    /* a pointer misses its alignment rule     */
#define MXS_ERR_UNSUPPORTED 3   /* size beyond a documented limit           */
#define MXS_ERR_CUDA 4          /* a CUDA call or launch failed             */
#define MXS_ERR_WORKSPACE 5     /* workspace NULL or smaller than required  */

/* Device-side condition bits written to *dev_status. */
#define MXS_DEV_BAD_DRAFT 0x1       /* spec_accept: a draft id outside [0,V)          */
#define MXS_DEV_ZERO_Q 0x2          /* spec_accept: a proposal with q(x) = 0 (reject) */
#define MXS_DEV_ZERO_RESIDUAL 0x4   /* spec_accept: residual mass 0, sampled p_j      */
#define MXS_DEV_NO_LAW 0x8          /* spec_accept / laws: a law with no mass         */
#define MXS_DEV_NEAR_EDGE 0x10      /* spec_accept: u within 1e-5 of a CDF bin edge   */
#define MXS_DEV_NONFINITE 0x20      /* mxfp4_pack: a block held Inf or NaN            */
#define MXS_DEV_TIMEOUT 0x40        /* a bounded pipeline wait gave up                */
#define MXS_DEV_KV_FULL 0x80        /* mxfp4_kv_append: a row fell past the cache     */

/* Input element types for mxfp4_pack. */
#define MXS_F32 0
#define MXS_BF16 1

/* ------------------------------------------------------------------------
 * mxfp4_pack
 *
 * Quantises real weights W [N, K] into the MXFP4 format used by
 * mxfp4_verify_gemm.  Format ("Module 11. Speculative Decoding and
 * Quantization", §12; "Next-Gen Speculative Decoding and FP4 Quantization
 * Shake Up LLM Inference Economics", section "Microscaling FP4 (MX-FP4)
 * Integration"): each run of 32 consecutive elements along K shares one E8M0
 * scale byte e (value 2^(e-127)); each element is a 4-bit E2M1 code
 * (sign | 2 exponent bits, bias 1 | 1 fraction bit; magnitudes
 * 0,0.5,1,1.5,2,3,4,6), two codes per byte, element k in byte k/2 with even
 * k in the low nibble.
 *
 * Rule per block: amax = max |w|; e_unb = the smallest integer with
 * amax <= 6 * 2^e_unb, clamped to [-127, 127] (no element is clipped);
 * an all-zero block gets e_unb = 0 (scale 1).  Each element becomes the
 * E2M1 value nearest to w / 2^e_unb, ties to the even fraction bit, with the
 * sign bit of w kept (so -0.0 and small negatives give code 8).
 *
 *   w        device, [N, K] fp32 (w_dtype MXS_F32) or bf16 (MXS_BF16),
 *            4- or 2-byte aligned
 *   nibbles  device, [N, K/2] uint8, written
 *   scales   device, [N, K/32] uint8, written
 *   N >= 0, K >= 0, K % 32 == 0
 * A block holding Inf or NaN gets scale byte 255 and zero nibbles and sets
 * MXS_DEV_NONFINITE.
 * ---------------------------------------------------------------------- */
mxs_status mxfp4_pack(const void* w, int32_t w_dtype, int64_t N, int64_t K,
                      uint8_t* nibbles, uint8_t* scales, int32_t* dev_status,
                      void* stream);

/* ------------------------------------------------------------------------
 * mxfp4_verify_gemm
 *
 * The weight-streaming GEMM of the verification pass: Y = X . dequant(W)^T,
 *   Y[m, n] = sum_k x[m, k] * e2m1(W[n, k]) * 2^(S[n, k/32] - 127),
 * with M = batch * (K_spec + 1) candidate positions ("Module 11 ...", §10:
 * verification as a short, wider decode; the fp32 accumulation and the
 * [rows, K/2] / [rows, K/32] layouts follow the MX-FP4 GEMV of "Next-Gen
 * Speculative Decoding and FP4 Quantization ...").
 *
 *   x          device, [M, K] bf16 (raw bits as uint16), 2-byte aligned
 *   nibbles    device, [N, K/2] uint8, 16-byte aligned
 *   scales     device, [N, K/32] uint8 (any alignment; copied to the
 *              workspace first when K % 512 != 0 or not 16-byte aligned)
 *   y          device, [M, N] fp32, 4-byte aligned, written
 *   1 <= M <= 65536, 1 <= N <= 4194240, 32 <= K <= 1048576, K % 32 == 0;
 *              rows are processed in passes of at most 32 or 64 (by the
 *              kernel, below), each pass one stream over W
 *   workspace  device, >= mxfp4_verify_gemm_workspace_size(M, N, K) bytes,
 *              16-byte aligned; scratch for the converted X, the split-K
 *              counters (zeroed by the call itself) and, when needed, the
 *              realigned scales.  Two calls in flight at the same time must
 *              not share a workspace.  The scales need no workspace copy when
 *              K % 512 == 0 and `scales` is 16-byte aligned; with K % 512 == 0
 *              a misaligned `scales` is rejected (MXS_ERR_MISALIGNED) because
 *              the size query assumed the in-place layout.
 *
 * Kernels and accuracy.  Products are exact and sums are fp32 in every path;
 * what differs is the image of x the tensor cores multiply:
 *   - passes of at most 8 rows: mma.sync on fp16 (each x row scaled by a
 *     power of two that puts its largest |x| in [2^15, 2^16): exact for every
 *     element within 2^29 of it), each 32-k block summed and scaled by its
 *     E8M0 factor in fp32, split-K when N is small;
 *   - passes of 9..32 rows: tcgen05 block-scaled MMA (kind::mxf4) on the E2M1
 *     weights and x as six E2M1 terms per 32-k block, each with its own
 *     power-of-two factor: x to within max|x| / 4^6 of each block maximum;
 *   - passes of 33..64 rows (K % 128 == 0): tcgen05 block-scaled MMA
 *     (kind::mxf8f6f4) with x as two E4M3 terms per 32-k block: exact for
 *     every element within 2^16 of its block maximum.
 * The paths add in different orders, so their results differ in the last
 * bits, all within the stated 2e-3 per-row bar (measured <= 1e-6 of each
 * row's largest output).  A row of x holding Inf or NaN gives a row of NaN.
 * MXS_GEMM_PATH=mma, bs4, bs8 or umma (an earlier tcgen05 kind::f16 kernel)
 * in the environment forces one kernel wherever it applies.
 * ---------------------------------------------------------------------- */
size_t mxfp4_verify_gemm_workspace_size(int64_t M, int64_t N, int64_t K);

mxs_status mxfp4_verify_gemm(const void* x, const uint8_t* nibbles,
                             const uint8_t* scales, float* y, int64_t M,
                             int64_t N, int64_t K, void* workspace,
                             size_t workspace_bytes, int32_t* dev_status,
                             void* stream);

/* ------------------------------------------------------------------------
 * mxfp4_verify_gemm_w4a4 -- the verify GEMM with MX-FP4 activations (W4A4)
 *
 * "Module 11. Speculative Decoding and Quantization", §12 ("Microscaled FP4,
 * W4A4, and the role of hardware"): weights and activations both MX-FP4.
 * Each 32-element block of each row of X is quantised by mxfp4_pack's rule
 * (e the smallest integer with max|x| <= 6 * 2^e, clamped to [-127, 127],
 * 0 for an all-zero block; each element the nearest E2M1 value of x / 2^e,
 * ties to the even code, the sign kept), and
 *   Y[m, n] = sum_k q(X)[m, k] * dequant(W)[n, k]     (fp32 accumulation).
 * This is a different product from mxfp4_verify_gemm's (X is rounded to 4
 * bits); the block-scaled tensor core takes both operands as stored, and a
 * pass covers up to 256 rows of X, so W is read once for M <= 256 (more
 * rows: as few passes as that allows, of equal size).
 *
 *   x, nibbles, scales, y, M, N, K: as for mxfp4_verify_gemm
 *   workspace  device, >= mxfp4_verify_gemm_w4a4_workspace_size(M, N, K)
 *              bytes, 16-byte aligned; not shared by two calls in flight
 * A row of X holding Inf or NaN gives NaN in every output of that row.
 * ---------------------------------------------------------------------- */
size_t mxfp4_verify_gemm_w4a4_workspace_size(int64_t M, int64_t N, int64_t K);

mxs_status mxfp4_verify_gemm_w4a4(const void* x, const uint8_t* nibbles,
                                  const uint8_t* scales, float* y, int64_t M,
                                  int64_t N, int64_t K, void* workspace,
                                  size_t workspace_bytes, int32_t* dev_status,
                                  void* stream);

/* ------------------------------------------------------------------------
 * nvfp4_verify_gemm -- the verify GEMM on NVFP4 weights
 *
 * Format ("Module 11. Speculative Decoding and Quantization", §12, NVFP4):
 * E2M1 codes as for MXFP4 (element k of row n in byte k/2 of [N, K/2], even k
 * in the low nibble), but each run of 16 consecutive elements along K shares
 * one E4M3 scale byte (sign | 4 exponent bits, bias 7 | 3 fraction bits;
 * subnormals at exponent field 0; 0x7F and 0xFF are NaN; largest finite 448),
 * and the whole tensor one FP32 scale g:
 *   Y[m, n] = g * sum_k x[m, k] * e2m1(W[n, k]) * e4m3(S[n, k/16]).
 *
 *   x            device, [M, K] bf16 (raw bits as uint16), 2-byte aligned
 *   nibbles      device, [N, K/2] uint8, 16-byte aligned
 *   scales       device, [N, K/16] uint8 E4M3 (any alignment; copied to the
 *                workspace first when K % 256 != 0 or not 16-byte aligned;
 *                with K % 256 == 0 a misaligned `scales` is rejected,
 *                MXS_ERR_MISALIGNED)
 *   global_scale the tensor's FP32 scale g, applied to every output
 *   y            device, [M, N] fp32, 4-byte aligned, written
 *   sizes        as for mxfp4_verify_gemm (K % 32 == 0)
 *   workspace    device, >= nvfp4_verify_gemm_workspace_size(M, N, K) bytes,
 *                16-byte aligned; not shared by two calls in flight
 *
 * Kernels and accuracy (products exact, sums fp32 in both):
 *   - passes of up to 64 rows: tcgen05 block-scaled MMA
 *     (kind::mxf4nvf4, scale_vec::4X) on the E2M1 codes with each scale
 *     read as UE4M3 (a negative scale is folded into its block's codes, a
 *     NaN scale gives NaN in its row n), and x as four E2M1 terms per 16-k
 *     block with UE4M3 factors: within ~1e-4 of each row's largest output
 *     on the parity cases, inside the 2e-3 bar;
 *   - MXS_GEMM_PATH=mma: passes of up to 64 rows on the mma.sync kernel,
 *     each decoded E2M1 code multiplied by its block's E4M3 scale in fp16
 *     (exact: at most 6 significant bits, in [2^-10, 2688]), x exact within
 *     2^29 of its row maximum.
 * Both apply g once, to the fp32 sum.  A row of x holding Inf or NaN gives a
 * row of NaN.
 * ---------------------------------------------------------------------- */
size_t nvfp4_verify_gemm_workspace_size(int64_t M, int64_t N, int64_t K);

mxs_status nvfp4_verify_gemm(const void* x, const uint8_t* nibbles,
                             const uint8_t* scales, float global_scale,
                             float* y, int64_t M, int64_t N, int64_t K,
                             void* workspace, size_t workspace_bytes,
                             int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * MX-FP4 KV cache of the verification block
 *
 * Keys and values stored as MX-FP4 ("Next-Gen Speculative Decoding and FP4
 * Quantization ...": the "KV Cache Memory Pool (FP4)" of its pipeline
 * diagram, "Benchmarks and Real-World Impact" item 2), and the unaccepted
 * suffix's entries discarded after acceptance ("Module 11 ...", §4).
 *
 * One cache holds one layer's keys (or values) for B sequences: nibbles
 * [B, L, W/2] and E8M0 scales [B, L, W/32] uint8, one row of W values (all
 * heads of one position, W % 32 == 0) per position, in the mxfp4_pack format;
 * lens [B] int32 (device) holds each sequence's committed length.
 *
 * mxfp4_kv_append: the verification pass feeds T = K + 1 positions per
 * sequence (the last committed token, then the K drafts).  Row t of
 * kv [B, T, W] (fp32 or bf16 by kv_dtype, 16-byte aligned) is packed by the
 * mxfp4_pack rule into position lens[b] + t.  Positions outside [0, L) are
 * not written and set MXS_DEV_KV_FULL; a non-finite block sets
 * MXS_DEV_NONFINITE.  lens is read, not changed.
 *
 * spec_kv_commit: lens[b] <- min(lens[b] + max(n_emitted[b], 0), L), with
 * n_emitted as spec_accept writes it.  The entries of the last committed
 * token and of the accepted drafts stay; the rejected drafts' entries are
 * the discarded suffix (overwritten by the next append); the replacement or
 * bonus token is fed, and cached, by the next pass.  A refused row (0
 * tokens) commits nothing.
 *
 * mxfp4_kv_dequant: out [B, L, W] fp32 (16-byte aligned) = the decoded
 * cache, exact, and 0 at every position l >= lens[b].
 *
 * Sizes: B, T >= 0, L >= 1, W >= 32, W % 32 == 0, B * L * W < 2^40.
 * ---------------------------------------------------------------------- */
mxs_status mxfp4_kv_append(const void* kv, int32_t kv_dtype, int64_t B, int64_t T,
                           int64_t W, uint8_t* nibbles, uint8_t* scales, int64_t L,
                           const int32_t* lens, int32_t* dev_status, void* stream);

mxs_status spec_kv_commit(int32_t* lens, const int32_t* n_emitted, int64_t B,
                          int64_t L, void* stream);

mxs_status mxfp4_kv_dequant(const uint8_t* nibbles, const uint8_t* scales,
                            int64_t B, int64_t L, int64_t W,
                            const int32_t* lens, float* out, void* stream);

/* ------------------------------------------------------------------------
 * mxfp4_verify_gemm_grouped -- many independent verify GEMMs in one go
 *
 * The verification pass runs every weight matrix of the target model over
 * the same M candidate positions ("Module 11 ...", §10).  When several of
 * those GEMMs are independent (Q, K, V or gate and up projections of one
 * layer, or any set whose outputs feed none of the others' inputs), one
 * grouped call converts each distinct X once and streams all of their
 * weights through persistent kernels, instead of paying two launches and a
 * pipeline fill per GEMM.
 *
 *   problems   HOST array of `count` descriptors, read during the call only.
 *              Per problem: x [M, K] bf16 (problems may share the same x),
 *              nibbles [N, K/2] (16-byte aligned), scales [N, K/32]
 *              (16-byte aligned, K % 512 == 0), y [M, N] fp32 written.
 *              No y may overlap any problem's x, nibbles, scales or another y.
 *   1 <= count <= 4096, 1 <= M <= 65536 (rows are processed in passes of at
 *   most 32 or 64, each pass one stream over every weight matrix)
 *   workspace  device, >= mxfp4_verify_gemm_grouped_workspace_size(...)
 *              bytes, 16-byte aligned.
 * Results are bit-identical to calling mxfp4_verify_gemm on each problem
 * whenever both take the same kernel and the single call does not split K
 * (splitting changes only the order of fp32 additions).  Both take the same
 * kernel for a pass of the same rows (one kind for every problem of a pass).
 * Within each mma.sync launch the problems are ordered by K, largest first,
 * and the CTAs claim work items (a 64- or 128-row tile) from a counter in
 * the workspace, zeroed by the call itself: a longest-first list schedule.
 * Every output element is still summed by one item in a fixed order, so the
 * results do not depend on which SM takes which item (MXS_GEMM_SCHED=static
 * selects a fixed round robin, for comparison).
 * ---------------------------------------------------------------------- */
typedef struct mxs_gemm_problem {
    const void* x;
    const uint8_t* nibbles;
    const uint8_t* scales;
    float* y;
    int64_t N;
    int64_t K;
} mxs_gemm_problem;

size_t mxfp4_verify_gemm_grouped_workspace_size(const mxs_gemm_problem* problems,
                                                int32_t count, int64_t M);

mxs_status mxfp4_verify_gemm_grouped(const mxs_gemm_problem* problems,
                                     int32_t count, int64_t M, void* workspace,
                                     size_t workspace_bytes,
                                     int32_t* dev_status, void* stream);

/* mxfp4_verify_gemm_grouped_w4a4 -- the grouped form of mxfp4_verify_gemm_w4a4
 * (W4A4, "Module 11 ...", §12): each distinct x is quantised to MX-FP4 by the
 * pack rule once per pass, and every weight matrix is streamed once per pass
 * of up to 256 rows.  Same problems, limits, errors and workspace rules as
 * mxfp4_verify_gemm_grouped (with its own workspace size); K is never split,
 * so each problem's result is bit-identical to mxfp4_verify_gemm_w4a4 on it
 * whenever that single call does not split K either. */
size_t mxfp4_verify_gemm_grouped_w4a4_workspace_size(const mxs_gemm_problem* problems,
                                                     int32_t count, int64_t M);

mxs_status mxfp4_verify_gemm_grouped_w4a4(const mxs_gemm_problem* problems,
                                          int32_t count, int64_t M, void* workspace,
                                          size_t workspace_bytes,
                                          int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * mxfp4_verify_gemm_noalloc -- the same GEMM for callers that cannot
 * allocate device memory.  (The pages have no counterpart: this is an
 * interface addition, not part of the method.)
 *
 * mxfp4_verify_gemm needs a workspace from its caller.  Some callers cannot
 * provide one: a plugin inside a host framework that owns every device
 * allocation and offers no scratch allocator, or a latency-critical path
 * where cudaMalloc's implicit device-wide synchronisation is not acceptable.
 * This entry point allocates nothing: its scratch is a file-scope device
 * array of MXS_NOALLOC_SCRATCH_BYTES (16 MiB) that every GPU loading this
 * part of the library holds until the process exits.
 *
 *   Arguments, layouts and accuracy as for mxfp4_verify_gemm, minus the
 *   workspace.  A shape whose scratch need
 *   (mxfp4_verify_gemm_workspace_size) exceeds MXS_NOALLOC_SCRATCH_BYTES is
 *   rejected with MXS_ERR_WORKSPACE before any launch.
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current) and caches it; make
 *   that first call before any stream capture.
 *   All calls on a device share the one array and it keeps the last call's
 *   contents (the kernels clear what must start at zero).  Calls that
 *   overlap on the GPU -- on different streams, or from different host
 *   threads -- race on it and must not be issued.
 * ---------------------------------------------------------------------- */
#define MXS_NOALLOC_SCRATCH_BYTES (16u << 20)

mxs_status mxfp4_verify_gemm_noalloc(const void* x, const uint8_t* nibbles,
                                     const uint8_t* scales, float* y,
                                     int64_t M, int64_t N, int64_t K,
                                     int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * spec_accept
 *
 * Exact speculative acceptance for B sequences with K draft tokens each
 * ("Module 11. Speculative Decoding and Quantization", §4 and §5):
 *   for i = 0..K-1: accept draft x_i while u[b,i] * q_i(x_i) < p_i(x_i)
 *   (the real-number comparison, exact; q_i(x_i) = 0 is a rejection);
 *   at the first rejection j sample the replacement from the residual
 *   r = (p_j - q_j)+ / sum (p_j - q_j)+, or, when all K were accepted
 *   (j = K), sample the bonus token from p_K.  The sample uses u[b,K] by
 *   inverse CDF: the smallest t with r_t > 0 and prefix_t > u[b,K] * S.
 *   Emits draft x_0..x_{j-1} and the sampled token; n_emitted = j + 1.
 *
 *   p           device, [B, K+1, V] fp32, target laws (p[b,K] = bonus law)
 *   q           device, [B, K, V] fp32, draft laws
 *   draft       device, [B, K] int32, draft token ids
 *   u           device, [B, K+1] fp32, uniforms in [0, 1)
 *   out_tokens  device, [B, K+1] int32, written, -1 after the last token
 *   n_emitted   device, [B] int32, written (0 for an error row)
 *   row_flags   device, [B] int32 or NULL: per-row MXS_DEV_* bits
 *   1 <= B < 2^31, 0 <= K <= 32, 1 <= V <= 2^21
 * Laws are used as given, never renormalised.  A row whose draft ids are not
 * all in [0, V) is an error row (n_emitted 0, tokens -1, MXS_DEV_BAD_DRAFT).
 * A residual with no mass falls back to p_j (MXS_DEV_ZERO_RESIDUAL); a law
 * with no finite positive mass gives an error row (MXS_DEV_NO_LAW).
 * MXS_DEV_NEAR_EDGE marks rows whose u[b,K] lay within 1e-5 (relative to S)
 * of an edge of the chosen bin, where the fp32 inputs' rounding may decide
 * the token.
 * ---------------------------------------------------------------------- */
mxs_status spec_accept(const float* p, const float* q, const int32_t* draft,
                       const float* u, int64_t B, int64_t K, int64_t V,
                       int32_t* out_tokens, int32_t* n_emitted,
                       int32_t* row_flags, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * Sampling laws from logits ("Module 11 ...", §4 "The exact propose-verify-
 * correct cycle"): acceptance must use the laws tokens are actually sampled
 * from -- temperature, top-k and top-p applied to the target and the draft
 * alike; raw probabilities with a filtered law break the proof.
 *
 * For one row of logits l[0..V-1]:
 *   - temperature T > 0 divides the logits;
 *   - top-k (k >= 1 and k < V; 0 or >= V: off) keeps every token whose logit
 *     is at least the k-th largest (ties at the boundary kept);
 *   - top-p (0 < p < 1; 1: off) then keeps, from the most probable down, the
 *     tokens up to the first whose cumulative mass reaches p, and every token
 *     as probable as that one (ties kept);
 *   - the kept tokens get p_t = exp((l_t - max l) / T) / S, the others 0.
 * A logit of -inf is a masked token (probability 0).  A row with a NaN or
 * +inf logit, or with every logit -inf, has no law: all probabilities 0 and
 * MXS_DEV_NO_LAW.  Masses are summed in fixed point (2^-46 units) so that
 * the top-p cut is a deterministic function of the row; probabilities match
 * a double-precision evaluation to ~1e-6 relative, and the cut may differ
 * from it only where p lies within ~1e-6 of a cumulative mass.
 *
 *   mxs_sampling   HOST struct: temperature (> 0, finite), top_k (>= 0),
 *                  top_p (in (0, 1])
 * ---------------------------------------------------------------------- */
typedef struct mxs_sampling {
    float temperature;
    int32_t top_k;
    float top_p;
} mxs_sampling;

/* spec_sampling_law: the transformed laws of R logit rows.
 *   logits  device, [R, V] fp32, 4-byte aligned
 *   probs   device, [R, V] fp32, written (may not overlap logits)
 *   1 <= R <= 2^28, 1 <= V <= 131072 (below 128 rows a cluster of up to 8 CTAs
 *   holds each row; from 128 rows one CTA streams each row) */
mxs_status spec_sampling_law(const float* logits, int64_t R, int64_t V,
                             const mxs_sampling* sampling, float* probs,
                             int32_t* dev_status, void* stream);

/* spec_accept_logits: spec_accept on the transformed laws of logits, without
 * writing the laws out: per-row statistics of every logit row (16 bytes each,
 * in the workspace) are computed first, then the acceptance kernel forms each
 * probability it needs from a logit and its row's statistics.  Results are
 * bit-identical to spec_accept on spec_sampling_law's outputs.
 *   target_logits  device, [B, K+1, V] fp32 (row K: the bonus position)
 *   draft_logits   device, [B, K, V] fp32
 *   draft, u, out_tokens, n_emitted, row_flags: as for spec_accept
 *   workspace      device, >= spec_accept_logits_workspace_size(B, K) bytes,
 *                  16-byte aligned
 *   1 <= B, B * (2K + 1) <= 2^28, 0 <= K <= 32, 1 <= V <= 131072 */
size_t spec_accept_logits_workspace_size(int64_t B, int64_t K);

mxs_status spec_accept_logits(const float* target_logits, const float* draft_logits,
                              const int32_t* draft, const float* u, int64_t B,
                              int64_t K, int64_t V, const mxs_sampling* sampling,
                              void* workspace, size_t workspace_bytes,
                              int32_t* out_tokens, int32_t* n_emitted,
                              int32_t* row_flags, int32_t* dev_status,
                              void* stream);

/* ------------------------------------------------------------------------
 * mxs_hbm_read_probe -- measurement helper (not part of the method):
 * streams `bytes` (multiple of 16) from `src` and writes a checksum to
 * *sink (device uint64).  Used to report a read-only HBM roofline.
 * ---------------------------------------------------------------------- */
mxs_status mxs_hbm_read_probe(const void* src, size_t bytes, uint64_t* sink,
                              void* stream);

/* ------------------------------------------------------------------------
 * mxs_hbm_copy_probe -- measurement helper (not part of the method): copies
 * `bytes` (multiple of 16) from `src` to `dst` (device, 16-byte aligned, not
 * overlapping).  Used for the read + write HBM roofline that the verify
 * GEMM's bandwidth is reported against.
 * ---------------------------------------------------------------------- */
mxs_status mxs_hbm_copy_probe(void* dst, const void* src, size_t bytes, void* stream);

/* Human-readable name of a status code (static string). */
const char* mxs_status_string(mxs_status status);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t mxs_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MXS_H_ */
