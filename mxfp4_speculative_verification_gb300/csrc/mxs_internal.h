// Host-side launchers behind the C ABI.  Arguments are validated by the
// entry points in api.cu before any of these is called.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace mxs {

// ---------------------------------------------------------------- GEMM
// Largest number of X rows handled by one pass over W (8 tiles of 8).
constexpr int kGemmMaxRowsPerPass = 64;

struct GemmWorkspace {
    size_t bytes;        // total
    size_t xf_off;       // fragment-ordered fp16 X, kGemmMaxRowsPerPass rows max
    size_t xun_off;      // per-row unscale factors (fp32)
    size_t cnt_off;      // split-K arrival counters (int32)
    int n_counters;
    size_t part_off;     // split-K partial tiles (fp32)
    size_t sc_off;       // realigned scales (only when needed)
    int sc_pitch;        // bytes per realigned scale row
    bool repack_scales;  // scales must be copied to the workspace first
};

// sdiv: k per scale byte, 32 (MXFP4) or 16 (NVFP4)
GemmWorkspace gemm_workspace_layout(int64_t M, int64_t N, int64_t K, bool scales_aligned, int sdiv = 32);

cudaError_t gemm_run(const uint16_t* x, const uint8_t* nibbles, const uint8_t* scales, float* y,
                     int64_t M, int64_t N, int64_t K, void* workspace,
                     const GemmWorkspace& ws, int32_t* dev_status, cudaStream_t stream);

// The same GEMM on NVFP4 weights: scales [N, K/16] E4M3, one FP32 tensor scale.
// W4A4: X quantised by the pack rule, passes of up to 256 rows (block-scaled kind::mxf4, one term)
GemmWorkspace gemm_w4a4_workspace_layout(int64_t M, int64_t N, int64_t K, bool scales_aligned);
cudaError_t gemm_run_w4a4(const uint16_t* x, const uint8_t* nibbles, const uint8_t* scales, float* y, int64_t M,
                          int64_t N, int64_t K, void* workspace, const GemmWorkspace& ws, int32_t* dev_status,
                          cudaStream_t stream);
cudaError_t gemm_run_nv(const uint16_t* x, const uint8_t* nibbles, const uint8_t* scales, float global_scale,
                        float* y, int64_t M, int64_t N, int64_t K, void* workspace, const GemmWorkspace& ws,
                        int32_t* dev_status, cudaStream_t stream);

// MX-FP4 KV cache of the verification block (kv.cu).
cudaError_t kv_append_run(const void* kv, int kv_dtype, int64_t B, int64_t T, int64_t W, uint8_t* nibbles,
                          uint8_t* scales, int64_t L, const int32_t* lens, int32_t* dev_status, cudaStream_t stream);
cudaError_t kv_commit_run(int32_t* lens, const int32_t* n_emitted, int64_t B, int64_t L, cudaStream_t stream);
cudaError_t kv_dequant_run(const uint8_t* nibbles, const uint8_t* scales, int64_t B, int64_t L, int64_t W,
                           const int32_t* lens, float* out, cudaStream_t stream);

// One GEMM of a grouped call (independent GEMMs sharing M <= 64).
struct GroupedGemm {
    const uint16_t* x;
    const uint8_t* nibbles;
    const uint8_t* scales;
    float* y;
    int64_t N, K;
};

// w4a4: every pass quantises X to MX-FP4 (the pack rule) and runs the
// block-scaled kind::mxf4 kernel with one term, up to 256 rows a pass
size_t gemm_grouped_workspace(const GroupedGemm* gs, int count, int64_t M, bool w4a4 = false);

cudaError_t gemm_grouped_run(const GroupedGemm* gs, int count, int64_t M, void* workspace,
                             int32_t* dev_status, cudaStream_t stream, bool w4a4 = false);

// ---------------------------------------------------------- acceptance
constexpr int kAcceptMaxK = 32;
constexpr int64_t kAcceptMaxV = int64_t(1) << 21;

cudaError_t accept_run(const float* p, const float* q, const int32_t* draft, const float* u,
                       int64_t B, int64_t K, int64_t V, int32_t* out_tokens,
                       int32_t* n_emitted, int32_t* row_flags, int32_t* dev_status,
                       cudaStream_t stream);

// ---------------------------------------------------- sampling laws
struct LawStats;
constexpr int64_t kLawMaxV = int64_t(1) << 17;  // 131072: a row per cluster of 8 CTAs, in registers

struct LawSampling {
    float temperature;  // > 0
    int64_t top_k;      // 0 (or >= V): off
    float top_p;        // (0, 1]; 1: off
};

// The transformed laws of R logit rows, written out ([R, V] fp32).
cudaError_t sampling_law_run(const float* logits, int64_t R, int64_t V, const LawSampling& s, float* probs,
                             int32_t* dev_status, cudaStream_t stream);
// Their per-row statistics only (`stats` holds R entries of 16 bytes).
cudaError_t law_stats_run(const float* logits, int64_t R, int64_t V, const LawSampling& s, LawStats* stats,
                          int32_t* dev_status, cudaStream_t stream);
// Both tensors' rows in one launch: stats[0 .. Ra) from logits_a, then stats[Ra .. Ra+Rb) from logits_b.
cudaError_t law_stats_run2(const float* logits_a, int64_t Ra, const float* logits_b, int64_t Rb, int64_t V,
                           const LawSampling& s, LawStats* stats, int32_t* dev_status, cudaStream_t stream);
constexpr size_t kLawStatsBytes = 16;

// Acceptance on laws given as logits + per-row statistics (the kernels of
// accept.cu evaluate each probability on the fly).
cudaError_t accept_logits_run(const float* p_logits, const float* q_logits, const LawStats* pst,
                              const LawStats* qst, float inv_t, const int32_t* draft, const float* u,
                              int64_t B, int64_t K, int64_t V, int32_t* out_tokens, int32_t* n_emitted,
                              int32_t* row_flags, int32_t* dev_status, cudaStream_t stream);

// ---------------------------------------------------------------- pack
cudaError_t pack_run(const void* w, int w_dtype, int64_t N, int64_t K, uint8_t* nibbles,
                     uint8_t* scales, int32_t* dev_status, cudaStream_t stream);

// --------------------------------------------------------------- probe
cudaError_t hbm_read_probe_run(const void* src, size_t bytes, uint64_t* sink,
                               cudaStream_t stream);
cudaError_t hbm_copy_probe_run(void* dst, const void* src, size_t bytes, cudaStream_t stream);

}  // namespace mxs
