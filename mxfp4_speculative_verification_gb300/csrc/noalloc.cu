// mxfp4_verify_gemm_noalloc: the verify GEMM for callers that cannot
// allocate device memory.
//
// mxfp4_verify_gemm needs a caller-provided workspace (converted X
// fragments, split-K partial tiles and their counters, realigned scales).
// Some callers have no way to obtain one: a plugin inside a host framework
// that owns every device allocation and offers no scratch allocator, or a
// latency-critical path where cudaMalloc's implicit device-wide
// synchronisation is not acceptable.  This entry point runs the same kernels
// with the scratch in a file-scope device array of fixed size instead, so it
// allocates nothing.  The pages have no counterpart to it.
#include <mutex>

#include "mxs.h"
#include "mxs_internal.h"

namespace {

// The scratch.  Every GPU that loads this part of the library holds it until
// the process exits; every call on a device uses the same bytes.
__device__ __align__(256) uint8_t g_noalloc_scratch[MXS_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
void* scratch_address(int dev) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

bool is_aligned(const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

}  // namespace

extern "C" mxs_status mxfp4_verify_gemm_noalloc(const void* x, const uint8_t* nibbles,
                                                const uint8_t* scales, float* y, int64_t M,
                                                int64_t N, int64_t K, int32_t* dev_status,
                                                void* stream) {
    if (!x || !nibbles || !scales || !y) return MXS_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 32 || K % 32 != 0) return MXS_ERR_INVALID_ARG;
    if (M > 65536 || N > int64_t(65535) * 64 || K > (int64_t(1) << 20)) return MXS_ERR_UNSUPPORTED;
    if (!is_aligned(x, 2) || !is_aligned(nibbles, 16) || !is_aligned(y, 4) ||
        !is_aligned(dev_status, 4))
        return MXS_ERR_MISALIGNED;
    const bool sc_aligned = is_aligned(scales, 16);
    if (K % 512 == 0 && !sc_aligned) return MXS_ERR_MISALIGNED;
    const mxs::GemmWorkspace ws = mxs::gemm_workspace_layout(M, N, K, sc_aligned);
    if (ws.bytes > MXS_NOALLOC_SCRATCH_BYTES) return MXS_ERR_WORKSPACE;  // shape needs more scratch
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MXS_ERR_CUDA;
    void* scratch = scratch_address(dev);
    if (!scratch) return MXS_ERR_CUDA;
    const cudaError_t e = mxs::gemm_run(static_cast<const uint16_t*>(x), nibbles, scales, y, M, N,
                                        K, scratch, ws, dev_status,
                                        static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MXS_OK : MXS_ERR_CUDA;
}
