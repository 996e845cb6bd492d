"""The no-allocation verify GEMM (mxfp4_verify_gemm_noalloc).

Callers that cannot allocate device memory -- for instance a plugin inside a
host framework that owns every device allocation and offers no scratch
allocator -- use this variant, whose scratch is a fixed 16 MiB device array
inside the library.  It must give the same result as the workspace entry
point, call after call, since every call reuses (and must re-clear) the same
scratch.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

import workloads
from helpers import GEMM_REL_TOL, bf16_tensor_from_bits, cuda_or_skip, gemm_row_rel_err

pytestmark = pytest.mark.gpu

MXS_ERR_WORKSPACE = 5


def _noalloc_fn(L):
    fn = L.mxfp4_verify_gemm_noalloc
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    fn.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp, vp]
    fn.restype = ctypes.c_int32
    return fn


@pytest.mark.parametrize("M,N,K", [(5, 4096, 14336),   # split K: partial tiles + counters
                                   (20, 1000, 544),     # K % 512 != 0: realigned scales
                                   (80, 384, 4096)])    # two passes over W
def test_noalloc_matches_workspace_entry_point_twice(M, N, K):
    torch, mxs = cuda_or_skip()
    dev = torch.device("cuda:0")
    fn = _noalloc_fn(mxs.lib())
    nib_h, sc_h = workloads.mxfp4_weights(N, K, 118, 132, seed=M + N, tensor_id=0)
    x = bf16_tensor_from_bits(torch, workloads.bf16_normal(M, K, seed=M + N, tensor_id=1), dev)
    nib, sc = torch.from_numpy(nib_h).to(dev), torch.from_numpy(sc_h).to(dev)
    ref = mxs.mxfp4_verify_gemm(x, nib, sc)
    stream = torch.cuda.current_stream(dev).cuda_stream
    outs = []
    for _ in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
        st = fn(x.data_ptr(), nib.data_ptr(), sc.data_ptr(), y.data_ptr(), M, N, K, None, stream)
        assert st == 0, mxs.lib().mxs_status_string(st)
        outs.append(y)
    torch.cuda.synchronize()
    r = ref.cpu().numpy()
    for y in outs:
        err = gemm_row_rel_err(y.cpu().numpy(), r)
        assert np.all(err <= GEMM_REL_TOL), f"max rel err {err.max():.3e}"


def test_noalloc_rejects_shapes_beyond_its_scratch():
    torch, mxs = cuda_or_skip()
    fn = _noalloc_fn(mxs.lib())
    M, N, K = 64, 64, 262144  # the X fragments alone need 32 MiB
    assert mxs.mxfp4_verify_gemm_workspace_size(M, N, K) > (16 << 20)
    dev = torch.device("cuda:0")
    x = torch.zeros((M, K), dtype=torch.bfloat16, device=dev)
    nib = torch.zeros((N, K // 2), dtype=torch.uint8, device=dev)
    sc = torch.zeros((N, K // 32), dtype=torch.uint8, device=dev)
    y = torch.zeros((M, N), dtype=torch.float32, device=dev)
    st = fn(x.data_ptr(), nib.data_ptr(), sc.data_ptr(), y.data_ptr(), M, N, K, None,
            torch.cuda.current_stream(dev).cuda_stream)
    assert st == MXS_ERR_WORKSPACE
