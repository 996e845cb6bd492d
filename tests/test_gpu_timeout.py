"""The bounded waits of the verify GEMM run out without hanging the GPU.

Every mbarrier wait of the kernels gives up after a time limit, sets
MXS_DEV_TIMEOUT in the caller's status word and lets the CTA leave.  Here the
limit is set short (1 ms) and the mma.sync kernel's producer leaves one stage
out entirely -- no copy issued, no arrival, so nothing is left in flight --
which makes the consumers' wait for that stage run out.  The call returns,
reports the timeout, and the next normal call is correct.  Both settings are
test-only environment overrides read by the host launcher (off by default).
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import GEMM_REL_TOL, bf16_tensor_from_bits, cuda_or_skip, gemm_row_rel_err

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_the_next_call_is_correct(monkeypatch):
    torch, mxs = cuda_or_skip()
    dev = torch.device("cuda:0")
    M, N, K = 5, 64, 16384          # mma.sync, one 64-row tile, 32 stages of 512 k
    nib_h, sc_h = workloads.mxfp4_weights(N, K, 118, 132, seed=11)
    xb = workloads.bf16_normal(M, K, seed=11)
    x = bf16_tensor_from_bits(torch, xb, dev)
    nib, sc = torch.from_numpy(nib_h).to(dev), torch.from_numpy(sc_h).to(dev)

    monkeypatch.setenv("MXS_GEMM_PATH", "mma")
    monkeypatch.setenv("MXS_GEMM_SPLITS", "1")
    monkeypatch.setenv("MXS_GEMM_WAIT_LIMIT_NS", "1000000")
    monkeypatch.setenv("MXS_GEMM_TEST_SKIP_STAGE", "6")
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    mxs.mxfp4_verify_gemm(x, nib, sc, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & mxs.DEV_FLAGS["TIMEOUT"]

    monkeypatch.delenv("MXS_GEMM_TEST_SKIP_STAGE")
    monkeypatch.delenv("MXS_GEMM_WAIT_LIMIT_NS")
    status.zero_()
    y = mxs.mxfp4_verify_gemm(x, nib, sc, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    err = gemm_row_rel_err(y.cpu().numpy(), oracle.gemm(xb, nib_h, sc_h))
    assert np.all(err <= GEMM_REL_TOL)
