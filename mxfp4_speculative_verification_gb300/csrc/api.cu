// The C ABI of libmxs (declared in include/mxs.h): host-side validation,
// then the launchers in gemm.cu, accept.cu and pack.cu.
#include <climits>
#include <cmath>
#include <cstdint>
#include <vector>

#include "mxs.h"
#include "mxs_internal.h"

namespace {

constexpr int64_t kMaxM = 65536;
constexpr int64_t kMaxN = 65535 * 64;
constexpr int64_t kMaxK = 1 << 20;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

mxs_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MXS_OK : MXS_ERR_CUDA; }

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

bool grouped_valid(const mxs_gemm_problem* problems, int32_t count, int64_t M,
                          std::vector<mxs::GroupedGemm>& out, mxs_status& st) {
    st = MXS_OK;
    if (!problems || count < 1 || M < 1) { st = MXS_ERR_INVALID_ARG; return false; }
    if (count > 4096 || M > kMaxM) { st = MXS_ERR_UNSUPPORTED; return false; }
    out.resize(size_t(count));
    for (int32_t i = 0; i < count; ++i) {
        const mxs_gemm_problem& p = problems[i];
        if (!p.x || !p.nibbles || !p.scales || !p.y || p.N < 1 || p.K < 32 || p.K % 32 != 0) {
            st = MXS_ERR_INVALID_ARG;
            return false;
        }
        if (p.N > kMaxN || p.K > kMaxK || p.K % 512 != 0) { st = MXS_ERR_UNSUPPORTED; return false; }
        if (!aligned(p.x, 2) || !aligned(p.nibbles, 16) || !aligned(p.scales, 16) || !aligned(p.y, 4)) {
            st = MXS_ERR_MISALIGNED;
            return false;
        }
        out[size_t(i)] = mxs::GroupedGemm{static_cast<const uint16_t*>(p.x), p.nibbles, p.scales,
                                          p.y, p.N, p.K};
    }
    return true;
}

}  // namespace

extern "C" {

mxs_status mxfp4_pack(const void* w, int32_t w_dtype, int64_t N, int64_t K, uint8_t* nibbles,
                      uint8_t* scales, int32_t* dev_status, void* stream) {
    if (N < 0 || K < 0 || K % 32 != 0) return MXS_ERR_INVALID_ARG;
    if (w_dtype != MXS_F32 && w_dtype != MXS_BF16) return MXS_ERR_INVALID_ARG;
    if (N == 0 || K == 0) return MXS_OK;
    if (!w || !nibbles || !scales) return MXS_ERR_INVALID_ARG;
    if (N > (int64_t(1) << 40) / K) return MXS_ERR_UNSUPPORTED;
    if (!aligned(w, w_dtype == MXS_F32 ? 4 : 2) || !aligned(dev_status, 4))
        return MXS_ERR_MISALIGNED;
    return cuda_status(
        mxs::pack_run(w, w_dtype, N, K, nibbles, scales, dev_status, as_stream(stream)));
}

size_t mxfp4_verify_gemm_workspace_size(int64_t M, int64_t N, int64_t K) {
    if (M < 1 || N < 1 || K < 32 || K % 32 != 0 || M > kMaxM || N > kMaxN || K > kMaxK) return 0;
    // the in-place scale layout is assumed when K % 512 == 0
    return mxs::gemm_workspace_layout(M, N, K, true).bytes;
}

mxs_status mxfp4_verify_gemm(const void* x, const uint8_t* nibbles, const uint8_t* scales,
                             float* y, int64_t M, int64_t N, int64_t K, void* workspace,
                             size_t workspace_bytes, int32_t* dev_status, void* stream) {
    if (!x || !nibbles || !scales || !y) return MXS_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 32 || K % 32 != 0) return MXS_ERR_INVALID_ARG;
    if (M > kMaxM || N > kMaxN || K > kMaxK) return MXS_ERR_UNSUPPORTED;
    if (!aligned(x, 2) || !aligned(nibbles, 16) || !aligned(y, 4) || !aligned(dev_status, 4))
        return MXS_ERR_MISALIGNED;
    const bool sc_aligned = aligned(scales, 16);
    if (K % 512 == 0 && !sc_aligned) return MXS_ERR_MISALIGNED;
    const mxs::GemmWorkspace ws = mxs::gemm_workspace_layout(M, N, K, sc_aligned);
    if (!workspace || workspace_bytes < ws.bytes) return MXS_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return MXS_ERR_MISALIGNED;
    return cuda_status(mxs::gemm_run(static_cast<const uint16_t*>(x), nibbles, scales, y, M, N, K,
                                     workspace, ws, dev_status, as_stream(stream)));
}

size_t mxfp4_verify_gemm_w4a4_workspace_size(int64_t M, int64_t N, int64_t K) {
    if (M < 1 || N < 1 || K < 32 || K % 32 != 0 || M > kMaxM || N > kMaxN || K > kMaxK) return 0;
    // the in-place scale layout is assumed when K % 512 == 0
    return mxs::gemm_w4a4_workspace_layout(M, N, K, true).bytes;
}

mxs_status mxfp4_verify_gemm_w4a4(const void* x, const uint8_t* nibbles, const uint8_t* scales, float* y,
                                  int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                                  int32_t* dev_status, void* stream) {
    if (!x || !nibbles || !scales || !y) return MXS_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 32 || K % 32 != 0) return MXS_ERR_INVALID_ARG;
    if (M > kMaxM || N > kMaxN || K > kMaxK) return MXS_ERR_UNSUPPORTED;
    if (!aligned(x, 2) || !aligned(nibbles, 16) || !aligned(y, 4) || !aligned(dev_status, 4))
        return MXS_ERR_MISALIGNED;
    const bool sc_aligned = aligned(scales, 16);
    if (K % 512 == 0 && !sc_aligned) return MXS_ERR_MISALIGNED;
    const mxs::GemmWorkspace ws = mxs::gemm_w4a4_workspace_layout(M, N, K, sc_aligned);
    if (!workspace || workspace_bytes < ws.bytes) return MXS_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return MXS_ERR_MISALIGNED;
    return cuda_status(mxs::gemm_run_w4a4(static_cast<const uint16_t*>(x), nibbles, scales, y, M, N, K, workspace,
                                          ws, dev_status, as_stream(stream)));
}

size_t nvfp4_verify_gemm_workspace_size(int64_t M, int64_t N, int64_t K) {
    if (M < 1 || N < 1 || K < 32 || K % 32 != 0 || M > kMaxM || N > kMaxN || K > kMaxK) return 0;
    // the in-place scale layout is assumed when K % 256 == 0
    return mxs::gemm_workspace_layout(M, N, K, true, 16).bytes;
}

mxs_status nvfp4_verify_gemm(const void* x, const uint8_t* nibbles, const uint8_t* scales,
                             float global_scale, float* y, int64_t M, int64_t N, int64_t K,
                             void* workspace, size_t workspace_bytes, int32_t* dev_status,
                             void* stream) {
    if (!x || !nibbles || !scales || !y) return MXS_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 32 || K % 32 != 0) return MXS_ERR_INVALID_ARG;
    if (M > kMaxM || N > kMaxN || K > kMaxK) return MXS_ERR_UNSUPPORTED;
    if (!aligned(x, 2) || !aligned(nibbles, 16) || !aligned(y, 4) || !aligned(dev_status, 4))
        return MXS_ERR_MISALIGNED;
    const bool sc_aligned = aligned(scales, 16);
    if (K % 256 == 0 && !sc_aligned) return MXS_ERR_MISALIGNED;
    const mxs::GemmWorkspace ws = mxs::gemm_workspace_layout(M, N, K, sc_aligned, 16);
    if (!workspace || workspace_bytes < ws.bytes) return MXS_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return MXS_ERR_MISALIGNED;
    return cuda_status(mxs::gemm_run_nv(static_cast<const uint16_t*>(x), nibbles, scales, global_scale, y,
                                        M, N, K, workspace, ws, dev_status, as_stream(stream)));
}

static bool kv_sizes_ok(int64_t B, int64_t L, int64_t W) {
    return B >= 0 && L >= 1 && W >= 32 && W % 32 == 0 && B <= (int64_t(1) << 31) &&
           (B == 0 || L <= ((int64_t(1) << 40) / W) / B) && L <= INT32_MAX;
}

mxs_status mxfp4_kv_append(const void* kv, int32_t kv_dtype, int64_t B, int64_t T, int64_t W, uint8_t* nibbles,
                           uint8_t* scales, int64_t L, const int32_t* lens, int32_t* dev_status, void* stream) {
    if (kv_dtype != MXS_F32 && kv_dtype != MXS_BF16) return MXS_ERR_INVALID_ARG;
    if (T < 0 || !kv_sizes_ok(B, L, W)) return MXS_ERR_INVALID_ARG;
    if (T > (int64_t(1) << 20)) return MXS_ERR_UNSUPPORTED;
    if (B == 0 || T == 0) return MXS_OK;
    if (!kv || !nibbles || !scales || !lens) return MXS_ERR_INVALID_ARG;
    if (!aligned(kv, 16) || !aligned(lens, 4) || !aligned(dev_status, 4)) return MXS_ERR_MISALIGNED;
    return cuda_status(mxs::kv_append_run(kv, kv_dtype, B, T, W, nibbles, scales, L, lens, dev_status,
                                          as_stream(stream)));
}

mxs_status spec_kv_commit(int32_t* lens, const int32_t* n_emitted, int64_t B, int64_t L, void* stream) {
    if (B < 0 || L < 1 || L > INT32_MAX) return MXS_ERR_INVALID_ARG;
    if (B == 0) return MXS_OK;
    if (!lens || !n_emitted) return MXS_ERR_INVALID_ARG;
    if (!aligned(lens, 4) || !aligned(n_emitted, 4)) return MXS_ERR_MISALIGNED;
    return cuda_status(mxs::kv_commit_run(lens, n_emitted, B, L, as_stream(stream)));
}

mxs_status mxfp4_kv_dequant(const uint8_t* nibbles, const uint8_t* scales, int64_t B, int64_t L, int64_t W,
                            const int32_t* lens, float* out, void* stream) {
    if (!kv_sizes_ok(B, L, W)) return MXS_ERR_INVALID_ARG;
    if (B == 0) return MXS_OK;
    if (!nibbles || !scales || !lens || !out) return MXS_ERR_INVALID_ARG;
    if (!aligned(nibbles, 16) || !aligned(lens, 4) || !aligned(out, 16)) return MXS_ERR_MISALIGNED;
    return cuda_status(mxs::kv_dequant_run(nibbles, scales, B, L, W, lens, out, as_stream(stream)));
}

size_t mxfp4_verify_gemm_grouped_workspace_size(const mxs_gemm_problem* problems, int32_t count,
                                                int64_t M) {
    std::vector<mxs::GroupedGemm> gs;
    mxs_status st;
    if (!grouped_valid(problems, count, M, gs, st)) return 0;
    return mxs::gemm_grouped_workspace(gs.data(), count, M);
}

mxs_status mxfp4_verify_gemm_grouped(const mxs_gemm_problem* problems, int32_t count, int64_t M,
                                     void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                     void* stream) {
    std::vector<mxs::GroupedGemm> gs;
    mxs_status st;
    if (!grouped_valid(problems, count, M, gs, st)) return st;
    if (!aligned(dev_status, 4)) return MXS_ERR_MISALIGNED;
    const size_t need = mxs::gemm_grouped_workspace(gs.data(), count, M);
    if (!workspace || workspace_bytes < need) return MXS_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return MXS_ERR_MISALIGNED;
    return cuda_status(mxs::gemm_grouped_run(gs.data(), count, M, workspace, dev_status,
                                             as_stream(stream)));
}

size_t mxfp4_verify_gemm_grouped_w4a4_workspace_size(const mxs_gemm_problem* problems, int32_t count,
                                                     int64_t M) {
    std::vector<mxs::GroupedGemm> gs;
    mxs_status st;
    if (!grouped_valid(problems, count, M, gs, st)) return 0;
    return mxs::gemm_grouped_workspace(gs.data(), count, M, true);
}

mxs_status mxfp4_verify_gemm_grouped_w4a4(const mxs_gemm_problem* problems, int32_t count, int64_t M,
                                          void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                          void* stream) {
    std::vector<mxs::GroupedGemm> gs;
    mxs_status st;
    if (!grouped_valid(problems, count, M, gs, st)) return st;
    if (!aligned(dev_status, 4)) return MXS_ERR_MISALIGNED;
    const size_t need = mxs::gemm_grouped_workspace(gs.data(), count, M, true);
    if (!workspace || workspace_bytes < need) return MXS_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return MXS_ERR_MISALIGNED;
    return cuda_status(mxs::gemm_grouped_run(gs.data(), count, M, workspace, dev_status, as_stream(stream), true));
}

mxs_status spec_accept(const float* p, const float* q, const int32_t* draft, const float* u,
                       int64_t B, int64_t K, int64_t V, int32_t* out_tokens, int32_t* n_emitted,
                       int32_t* row_flags, int32_t* dev_status, void* stream) {
    if (B < 1 || K < 0 || V < 1) return MXS_ERR_INVALID_ARG;
    if (B > INT32_MAX || K > mxs::kAcceptMaxK || V > mxs::kAcceptMaxV) return MXS_ERR_UNSUPPORTED;
    if (!p || !u || !out_tokens || !n_emitted) return MXS_ERR_INVALID_ARG;
    if (K > 0 && (!q || !draft)) return MXS_ERR_INVALID_ARG;
    if (!aligned(p, 4) || !aligned(q, 4) || !aligned(draft, 4) || !aligned(u, 4) ||
        !aligned(out_tokens, 4) || !aligned(n_emitted, 4) || !aligned(row_flags, 4) ||
        !aligned(dev_status, 4))
        return MXS_ERR_MISALIGNED;
    return cuda_status(mxs::accept_run(p, q, draft, u, B, K, V, out_tokens, n_emitted, row_flags,
                                       dev_status, as_stream(stream)));
}

static bool sampling_ok(const mxs_sampling* s) {
    return s && s->temperature > 0.f && std::isfinite(s->temperature) && s->top_k >= 0 && s->top_p > 0.f &&
           s->top_p <= 1.f;
}

static mxs::LawSampling law_sampling(const mxs_sampling* s) {
    mxs::LawSampling l;
    l.temperature = s->temperature;
    l.top_k = s->top_k;
    l.top_p = s->top_p;
    return l;
}

mxs_status spec_sampling_law(const float* logits, int64_t R, int64_t V, const mxs_sampling* sampling,
                             float* probs, int32_t* dev_status, void* stream) {
    if (R < 1 || V < 1 || !logits || !probs || !sampling_ok(sampling)) return MXS_ERR_INVALID_ARG;
    if (V > mxs::kLawMaxV || R > INT32_MAX / 8) return MXS_ERR_UNSUPPORTED;
    if (!aligned(logits, 4) || !aligned(probs, 4) || !aligned(dev_status, 4)) return MXS_ERR_MISALIGNED;
    return cuda_status(mxs::sampling_law_run(logits, R, V, law_sampling(sampling), probs, dev_status,
                                             as_stream(stream)));
}

size_t spec_accept_logits_workspace_size(int64_t B, int64_t K) {
    if (B < 1 || K < 0 || K > mxs::kAcceptMaxK || B > INT32_MAX) return 0;
    return size_t(B) * size_t(2 * K + 1) * mxs::kLawStatsBytes;
}

mxs_status spec_accept_logits(const float* target_logits, const float* draft_logits, const int32_t* draft,
                              const float* u, int64_t B, int64_t K, int64_t V, const mxs_sampling* sampling,
                              void* workspace, size_t workspace_bytes, int32_t* out_tokens,
                              int32_t* n_emitted, int32_t* row_flags, int32_t* dev_status, void* stream) {
    if (B < 1 || K < 0 || V < 1 || !sampling_ok(sampling)) return MXS_ERR_INVALID_ARG;
    if (B > INT32_MAX || K > mxs::kAcceptMaxK || V > mxs::kLawMaxV || B * (2 * K + 1) > INT32_MAX / 8)
        return MXS_ERR_UNSUPPORTED;
    if (!target_logits || !u || !out_tokens || !n_emitted) return MXS_ERR_INVALID_ARG;
    if (K > 0 && (!draft_logits || !draft)) return MXS_ERR_INVALID_ARG;
    if (!aligned(target_logits, 4) || !aligned(draft_logits, 4) || !aligned(draft, 4) || !aligned(u, 4) ||
        !aligned(out_tokens, 4) || !aligned(n_emitted, 4) || !aligned(row_flags, 4) || !aligned(dev_status, 4))
        return MXS_ERR_MISALIGNED;
    const size_t need = spec_accept_logits_workspace_size(B, K);
    if (!workspace || workspace_bytes < need) return MXS_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return MXS_ERR_MISALIGNED;
    const cudaStream_t st = as_stream(stream);
    const mxs::LawSampling ls = law_sampling(sampling);
    mxs::LawStats* pst = static_cast<mxs::LawStats*>(workspace);
    mxs::LawStats* qst = reinterpret_cast<mxs::LawStats*>(static_cast<char*>(workspace) +
                                                          size_t(B) * size_t(K + 1) * mxs::kLawStatsBytes);
    // the target's and the draft's rows in one launch (qst follows pst)
    cudaError_t e = mxs::law_stats_run2(target_logits, B * (K + 1), draft_logits, B * K, V, ls, pst, dev_status, st);
    if (e == cudaSuccess)
        e = mxs::accept_logits_run(target_logits, draft_logits, pst, qst, 1.0f / sampling->temperature, draft,
                                   u, B, K, V, out_tokens, n_emitted, row_flags, dev_status, st);
    return cuda_status(e);
}

mxs_status mxs_hbm_read_probe(const void* src, size_t bytes, uint64_t* sink, void* stream) {
    if (!src || !sink || bytes == 0 || bytes % 16 != 0) return MXS_ERR_INVALID_ARG;
    if (!aligned(src, 16) || !aligned(sink, 8)) return MXS_ERR_MISALIGNED;
    return cuda_status(mxs::hbm_read_probe_run(src, bytes, sink, as_stream(stream)));
}

mxs_status mxs_hbm_copy_probe(void* dst, const void* src, size_t bytes, void* stream) {
    if (!dst || !src || bytes == 0 || bytes % 16 != 0) return MXS_ERR_INVALID_ARG;
    if (!aligned(src, 16) || !aligned(dst, 16)) return MXS_ERR_MISALIGNED;
    const char* d = static_cast<const char*>(dst);
    const char* sp = static_cast<const char*>(src);
    if (d < sp + bytes && sp < d + bytes) return MXS_ERR_INVALID_ARG;  // overlapping buffers
    return cuda_status(mxs::hbm_copy_probe_run(dst, src, bytes, as_stream(stream)));
}

const char* mxs_status_string(mxs_status status) {
    switch (status) {
        case MXS_OK: return "MXS_OK";
        case MXS_ERR_INVALID_ARG: return "MXS_ERR_INVALID_ARG";
        case MXS_ERR_MISALIGNED: return "MXS_ERR_MISALIGNED";
        case MXS_ERR_UNSUPPORTED: return "MXS_ERR_UNSUPPORTED";
        case MXS_ERR_CUDA: return "MXS_ERR_CUDA";
        case MXS_ERR_WORKSPACE: return "MXS_ERR_WORKSPACE";
        default: return "MXS_ERR_UNKNOWN";
    }
}

int32_t mxs_version(void) { return 100; }

}  // extern "C"
