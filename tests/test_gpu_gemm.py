"""GPU parity of mxfp4_verify_gemm against the CPU oracle.

Bar: per output row m, max_n |Y_gpu - Y_ref| / max_n |Y_ref| <= 2e-3, with
Y_ref the oracle's double-precision definition on the same seeded inputs.
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import GEMM_REL_TOL, bf16_tensor_from_bits, cuda_or_skip, gemm_row_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    return cuda_or_skip()


def _run(env, x_bits, nib, sc, **kw):
    torch, mxs = env
    dev = torch.device("cuda:0")
    x = bf16_tensor_from_bits(torch, x_bits, dev)
    y = mxs.mxfp4_verify_gemm(x, torch.from_numpy(nib).to(dev), torch.from_numpy(sc).to(dev), **kw)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def _check(env, x_bits, nib, sc, tol=GEMM_REL_TOL):
    y = _run(env, x_bits, nib, sc)
    ref = oracle.gemm(x_bits, nib, sc)
    err = gemm_row_rel_err(y, ref)
    assert np.all(err <= tol), f"max rel err {err.max():.3e}"
    return err.max()


def test_hand_worked_block(env):
    nib = np.zeros((1, 16), dtype=np.uint8)
    nib[0, 0] = 0x3A
    sc = np.array([[126]], dtype=np.uint8)
    x = workloads.f32_to_bf16_bits(np.array([[1.0, 2.0] + [0.0] * 30], dtype=np.float32))
    assert _run(env, x, nib, sc)[0, 0] == 1.0


def test_every_code_and_nibble_position(env):
    # row n holds code (n % 16) at every position: exercises the decode table
    # and the nibble order for all 16 codes in both halves of a byte
    K = 64
    codes = np.arange(16, dtype=np.uint8).repeat(K).reshape(16, K)
    nib = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sc = np.full((16, 2), 127, dtype=np.uint8)
    rng = np.random.default_rng(1)
    x = workloads.f32_to_bf16_bits(rng.standard_normal((3, K)).astype(np.float32))
    y = _run(env, x, nib, sc)
    assert np.array_equal(y.astype(np.float64), oracle.gemm(x, nib, sc)) or \
        np.all(gemm_row_rel_err(y, oracle.gemm(x, nib, sc)) < 1e-6)
    # one-hot positions: element k alone non-zero picks x[:, k]
    for k in (0, 1, 2, 31, 33, 63):
        c = np.zeros((1, K), dtype=np.uint8)
        c[0, k] = 3  # 1.5
        nb = (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
        yk = _run(env, x, nb, np.full((1, 2), 127, dtype=np.uint8))
        xv = (x.astype(np.uint32) << 16).view(np.float32)
        assert np.array_equal(yk[:, 0], 1.5 * xv[:, k])


def test_tiny_config(env):
    x, nib, sc = workloads.tiny_gemm_inputs(0)
    _check(env, x, nib, sc)


@pytest.mark.parametrize("M", [1, 2, 5, 8, 9, 16, 17, 20, 24, 32, 33, 40, 64, 65, 80])
def test_rows_m(env, M):
    nib, sc = workloads.mxfp4_weights(300, 1024, 118, 132, seed=M, tensor_id=0)
    x = workloads.bf16_normal(M, 1024, seed=M, tensor_id=1)
    _check(env, x, nib, sc)


@pytest.mark.parametrize("N,K", [(1, 32), (7, 64), (63, 512), (65, 544), (129, 1056),
                                 (200, 4096), (257, 2080), (1000, 14336), (130, 8192 + 32)])
def test_ragged_shapes(env, N, K):
    nib, sc = workloads.mxfp4_weights(N, K, 118, 132, seed=N + K, tensor_id=0)
    x = workloads.bf16_normal(5, K, seed=N + K, tensor_id=1)
    _check(env, x, nib, sc)


def test_split_k_cluster_path(env):
    # few rows, long K: the launcher splits K across a thread-block cluster
    nib, sc = workloads.mxfp4_weights(64, 28672, 118, 132, seed=3, tensor_id=0)
    x = workloads.bf16_normal(5, 28672, seed=3, tensor_id=1)
    _check(env, x, nib, sc)


def test_full_exponent_range(env):
    # E8M0 bytes 0..254 (2^-127 .. 2^127); values stay finite in fp32
    rng = np.random.default_rng(5)
    N, K = 64, 512
    nib = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sc = rng.integers(0, 200, size=(N, K // 32)).astype(np.uint8)
    sc[0, :] = 0
    sc[1, :] = 199
    x = workloads.bf16_normal(3, K, seed=5)
    _check(env, x, nib, sc)


def test_nan_scale(env):
    nib = np.full((2, 16), 0x22, dtype=np.uint8)
    sc = np.array([[255], [127]], dtype=np.uint8)
    x = workloads.f32_to_bf16_bits(np.ones((1, 32), dtype=np.float32))
    y = _run(env, x, nib, sc)
    assert np.isnan(y[0, 0]) and y[0, 1] == 32.0


@pytest.mark.parametrize("scale", [2.0 ** -120, 2.0 ** -30, 1e-3, 1e4, 3e4, 1e9, 2.0 ** 100])
def test_activation_magnitudes(env, scale):
    # X rows far outside fp16 range still match (power-of-two row scaling)
    nib, sc = workloads.mxfp4_weights(96, 512, 118, 132, seed=9)
    rng = np.random.default_rng(9)
    xf = (rng.standard_normal((4, 512)) * scale).astype(np.float32)
    xf[1] *= 1e-3
    x = workloads.f32_to_bf16_bits(xf)
    _check(env, x, nib, sc)


def test_zero_rows_and_zero_weights(env):
    nib, sc = workloads.mxfp4_weights(64, 512, 118, 132, seed=2)
    nib[5] = 0
    x = workloads.bf16_normal(3, 512, seed=2)
    x[1] = 0
    y = _run(env, x, nib, sc)
    assert np.all(y[1] == 0) and np.all(y[:, 5] == 0)


def test_deterministic_run_to_run(env):
    torch, mxs = env
    nib, sc = workloads.mxfp4_weights(512, 8192, 118, 132, seed=4)
    x = workloads.bf16_normal(5, 8192, seed=4)
    a = _run(env, x, nib, sc)
    b = _run(env, x, nib, sc)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("idx,name,K,N", [(i,) + s for i, s in
                                           enumerate(list(workloads.LLAMA8B_LAYER) + [workloads.LLAMA8B_LM_HEAD])])
def test_llama8b_layer_full(env, idx, name, K, N):
    nib, sc = workloads.mxfp4_weights(N, K, *workloads.LLAMA_EXP_RANGE, seed=0, tensor_id=100 + idx)
    x = workloads.bf16_normal(5, K, seed=0, tensor_id=7)
    _check(env, x, nib, sc)


@pytest.mark.parametrize("name,K,N", list(workloads.LLAMA70B_LAYER) + [workloads.LLAMA70B_LM_HEAD])
@pytest.mark.parametrize("M", [5, 20, 80])
def test_llama70b_layer_sampled_rows(env, name, K, N, M):
    """Full-size 70B layer on the device; 256 sampled output columns checked."""
    torch, mxs = env
    dev = torch.device("cuda:0")
    nib_d, sc_d = workloads.device_mxfp4_weights(N, K, *workloads.LLAMA_EXP_RANGE, seed=M, device=dev)
    x_d = workloads.device_bf16_normal(M, K, seed=M + 1, device=dev)
    y = mxs.mxfp4_verify_gemm(x_d, nib_d, sc_d)
    torch.cuda.synchronize()
    rng = np.random.default_rng(M)
    cols = np.sort(rng.choice(N, size=256, replace=False))
    cols[0], cols[-1] = 0, N - 1
    idx = torch.from_numpy(cols).to(dev)
    nib = nib_d.index_select(0, idx).cpu().numpy()
    sc = sc_d.index_select(0, idx).cpu().numpy()
    xb = x_d.view(torch.int16).cpu().numpy().view(np.uint16)
    ref = oracle.gemm(xb, nib, sc)
    got = y.index_select(1, idx).cpu().numpy()
    # per-row bar, with the reference max over the sampled columns
    err = gemm_row_rel_err(got, ref)
    assert np.all(err <= GEMM_REL_TOL), f"max rel err {err.max():.3e}"


def test_misaligned_scales_rejected_and_repacked(env):
    torch, mxs = env
    dev = torch.device("cuda:0")
    N, K = 64, 544  # K % 512 != 0: realigned through the workspace
    nib, sc = workloads.mxfp4_weights(N, K, 118, 132, seed=6)
    buf = torch.zeros(sc.size + 1, dtype=torch.uint8, device=dev)
    buf[1:] = torch.from_numpy(sc.ravel()).to(dev)
    sc_off = buf[1:].view(N, K // 32)  # 1 byte off 16-byte alignment
    x = workloads.bf16_normal(5, K, seed=6)
    y = mxs.mxfp4_verify_gemm(bf16_tensor_from_bits(torch, x, dev), torch.from_numpy(nib).to(dev), sc_off)
    torch.cuda.synchronize()
    assert np.all(gemm_row_rel_err(y.cpu().numpy(), oracle.gemm(x, nib, sc)) <= GEMM_REL_TOL)
    # with K % 512 == 0 the in-place layout is required
    N, K = 64, 512
    nib, sc = workloads.mxfp4_weights(N, K, 118, 132, seed=6)
    buf = torch.zeros(sc.size + 1, dtype=torch.uint8, device=dev)
    with pytest.raises(mxs.MxsError, match="MISALIGNED"):
        mxs.mxfp4_verify_gemm(bf16_tensor_from_bits(torch, workloads.bf16_normal(5, K, seed=6), dev),
                              torch.from_numpy(nib).to(dev), buf[1:].view(N, K // 32))


def test_no_timeout_reported(env):
    torch, mxs = env
    dev = torch.device("cuda:0")
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    nib, sc = workloads.mxfp4_weights(4096, 4096, 118, 132, seed=8)
    x = workloads.bf16_normal(5, 4096, seed=8)
    mxs.mxfp4_verify_gemm(bf16_tensor_from_bits(torch, x, dev), torch.from_numpy(nib).to(dev),
                          torch.from_numpy(sc).to(dev), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
