"""GPU parity of the tcgen05 (tensor memory) verify-GEMM path used for M > 24.

The entry points pick this path on their own only for wide passes (and, for
a single GEMM, wide outputs); here it is forced (MXS_GEMM_PATH=umma) so that
small, ragged and pathological shapes exercise it too, against the same
oracle and bar.
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import GEMM_REL_TOL, bf16_tensor_from_bits, cuda_or_skip, gemm_row_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture
def env(monkeypatch):
    monkeypatch.setenv("MXS_GEMM_PATH", "umma")
    return cuda_or_skip()


def _check(env, x, nib, sc):
    torch, mxs = env
    dev = torch.device("cuda:0")
    y = mxs.mxfp4_verify_gemm(bf16_tensor_from_bits(torch, x, dev), torch.from_numpy(nib).to(dev),
                              torch.from_numpy(sc).to(dev))
    torch.cuda.synchronize()
    ref = oracle.gemm(x, nib, sc)
    err = gemm_row_rel_err(y.cpu().numpy(), ref)
    assert np.all(err <= GEMM_REL_TOL), f"max rel err {err.max():.3e}"
    return y.cpu().numpy(), ref


@pytest.mark.parametrize("M", [9, 16, 17, 20, 32, 33, 48, 49, 64, 65, 80])
def test_umma_rows_m(env, M):
    nib, sc = workloads.mxfp4_weights(300, 1024, 118, 132, seed=M, tensor_id=0)
    x = workloads.bf16_normal(M, 1024, seed=M, tensor_id=1)
    _check(env, x, nib, sc)


@pytest.mark.parametrize("N,K", [(1, 32), (127, 512), (129, 544), (200, 4096), (257, 2080),
                                 (1000, 14336), (130, 8192 + 32)])
def test_umma_ragged(env, N, K):
    nib, sc = workloads.mxfp4_weights(N, K, 118, 132, seed=N + K, tensor_id=0)
    x = workloads.bf16_normal(20, K, seed=N + K, tensor_id=1)
    _check(env, x, nib, sc)


def test_umma_every_code(env):
    K = 64
    codes = np.arange(16, dtype=np.uint8).repeat(K).reshape(16, K)
    nib = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sc = np.full((16, 2), 127, dtype=np.uint8)
    x = workloads.bf16_normal(12, K, seed=1)
    y, ref = _check(env, x, nib, sc)
    assert np.all(gemm_row_rel_err(y, ref) < 1e-6)


@pytest.mark.parametrize("lo,hi", [(0, 200), (100, 140), (60, 61)])
def test_umma_exponent_spreads(env, lo, hi):
    # blocks more than 26 binades below their row's maximum take the exact CUDA-core route
    rng = np.random.default_rng(lo)
    N, K = 256, 1024
    nib = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sc = rng.integers(lo, hi + 1, size=(N, K // 32)).astype(np.uint8)
    sc[0, :] = lo
    x = workloads.bf16_normal(20, K, seed=lo)
    _check(env, x, nib, sc)


def test_umma_isolated_small_blocks(env):
    # one row with a single tiny block among large ones: its contribution must survive
    N, K = 128, 512
    codes = np.zeros((N, K), dtype=np.uint8)
    codes[:, :] = 7  # 6.0
    nib = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sc = np.full((N, K // 32), 160, dtype=np.uint8)
    sc[5, 3] = 100      # 60 binades below the row maximum
    sc[6, :] = 100
    sc[6, 9] = 130
    x = workloads.bf16_normal(16, K, seed=3)
    _check(env, x, nib, sc)


@pytest.mark.parametrize("N", [128, 300])
def test_umma_late_row_maximum(env, N):
    # each row's largest exponent sits in its last stage, 40 binades above the rest:
    # every earlier block of every row goes through the exact accumulator, across
    # several stages and (N = 300) several tiles per CTA
    K = 2048
    rng = np.random.default_rng(N)
    nib = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sc = np.full((N, K // 32), 100, dtype=np.uint8)
    sc[:, -16:] = 140
    sc[::3, 5] = 139
    x = workloads.bf16_normal(20, K, seed=N)
    _check(env, x, nib, sc)


def test_umma_nan_scale(env):
    nib = np.full((2, 16), 0x22, dtype=np.uint8)
    sc = np.array([[255], [127]], dtype=np.uint8)
    x = workloads.f32_to_bf16_bits(np.ones((12, 32), dtype=np.float32))
    torch, mxs = env
    dev = torch.device("cuda:0")
    y = mxs.mxfp4_verify_gemm(bf16_tensor_from_bits(torch, x, dev), torch.from_numpy(nib).to(dev),
                              torch.from_numpy(sc).to(dev)).cpu().numpy()
    assert np.all(np.isnan(y[:, 0])) and np.all(y[:, 1] == 32.0)


@pytest.mark.parametrize("scale", [2.0 ** -120, 1e-3, 3e4, 2.0 ** 100])
def test_umma_activation_magnitudes(env, scale):
    nib, sc = workloads.mxfp4_weights(160, 512, 118, 132, seed=9)
    rng = np.random.default_rng(9)
    xf = (rng.standard_normal((20, 512)) * scale).astype(np.float32)
    xf[1] *= 1e-3
    _check(env, workloads.f32_to_bf16_bits(xf), nib, sc)


def test_umma_deterministic_and_status_clean(env):
    torch, mxs = env
    dev = torch.device("cuda:0")
    nib, sc = workloads.mxfp4_weights(4096, 4096, 118, 132, seed=4)
    x = bf16_tensor_from_bits(torch, workloads.bf16_normal(40, 4096, seed=4), dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    a = mxs.mxfp4_verify_gemm(x, torch.from_numpy(nib).to(dev), torch.from_numpy(sc).to(dev),
                              dev_status=status)
    b = mxs.mxfp4_verify_gemm(x, torch.from_numpy(nib).to(dev), torch.from_numpy(sc).to(dev))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("idx,name,K,N", [(i,) + s for i, s in
                                           enumerate(list(workloads.LLAMA8B_LAYER) + [workloads.LLAMA8B_LM_HEAD])])
def test_umma_llama8b_layer_m40(env, idx, name, K, N):
    nib, sc = workloads.mxfp4_weights(N, K, *workloads.LLAMA_EXP_RANGE, seed=0, tensor_id=200 + idx)
    x = workloads.bf16_normal(40, K, seed=0, tensor_id=8)
    _check(env, x, nib, sc)
