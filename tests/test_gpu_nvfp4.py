"""GPU parity of nvfp4_verify_gemm against the CPU oracle ("Module 11.
Speculative Decoding and Quantization", §12, NVFP4: E2M1 values in blocks of
16 sharing an E4M3 scale, one FP32 scale per tensor).

Bar: per output row m, max_n |Y_gpu - Y_ref| / max_n |Y_ref| <= 2e-3 (the
verify GEMM's bar), Y_ref the oracle's double-precision definition on the same
seeded inputs.  Every test runs on both kernels: the mma.sync kernel (exact
products: the decode checks are exact or within 1e-6) and the block-scaled
tcgen05 kernel (X as four E2M1 terms: every check within 5e-4 of the row
maximum, four times inside the bar; a misread scale would be off by O(1)).
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import GEMM_REL_TOL, bf16_tensor_from_bits, cuda_or_skip, gemm_row_rel_err

pytestmark = pytest.mark.gpu

TOL = {"mma": 1e-5, "bs": 5e-4}


@pytest.fixture(scope="module")
def env():
    return cuda_or_skip()


@pytest.fixture(params=["mma", "bs"], autouse=True)
def path(request, monkeypatch):
    monkeypatch.setenv("MXS_GEMM_PATH", request.param)
    return request.param


def _run(env, x_bits, nib, sc, g=1.0, sc_offset=0, **kw):
    torch, mxs = env
    dev = torch.device("cuda:0")
    x = bf16_tensor_from_bits(torch, x_bits, dev)
    if sc_offset:
        # the same scale bytes at a misaligned address
        buf = torch.zeros(sc.size + sc_offset, dtype=torch.uint8, device=dev)
        buf[sc_offset:] = torch.from_numpy(sc.reshape(-1)).to(dev)
        t_sc = buf[sc_offset:].view(sc.shape)
    else:
        t_sc = torch.from_numpy(sc).to(dev)
    y = mxs.nvfp4_verify_gemm(x, torch.from_numpy(nib).to(dev), t_sc, g, **kw)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def _check(env, x_bits, nib, sc, g=1.0, tol=GEMM_REL_TOL, **kw):
    y = _run(env, x_bits, nib, sc, g, **kw)
    ref = oracle.nvfp4_gemm(x_bits, nib, sc, g)
    err = gemm_row_rel_err(y, ref)
    assert np.all(err <= tol), f"max rel err {err.max():.3e}"
    return err.max()


def _pack_codes(codes):
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def test_hand_worked_block(env, path):
    # codes 1.0 (2) and -3.0 (13) under scale 0x40 (= 2.0) and g = 0.5:
    # y = 0.5 * 2 * (1 * 1.0 + 2 * -3.0) = -5
    codes = np.zeros((1, 32), np.uint8)
    codes[0, 0], codes[0, 1] = 2, 13
    sc = np.array([[0x40, 0x38]], np.uint8)
    x = workloads.f32_to_bf16_bits(np.array([[1.0, 2.0] + [0.0] * 30], np.float32))
    y = _run(env, x, _pack_codes(codes), sc, 0.5)[0, 0]
    assert y == -5.0 if path == "mma" else abs(y + 5.0) <= 5.0 * TOL[path]


def test_every_e4m3_scale_byte(env, path):
    # row n: its first 16-element block under scale byte n, the second under
    # 1.0 (0x38); every E4M3 code including subnormals, negatives and NaN
    K = 32
    rng = np.random.default_rng(4)
    codes = rng.integers(0, 16, size=(256, K)).astype(np.uint8)
    sc = np.stack([np.arange(256, dtype=np.uint8), np.full(256, 0x38, np.uint8)], axis=1)
    x = workloads.f32_to_bf16_bits(rng.standard_normal((3, K)).astype(np.float32))
    y = _run(env, x, _pack_codes(codes), sc, 1.0)
    ref = oracle.nvfp4_gemm(x, _pack_codes(codes), sc, 1.0)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(y), nan) and set(np.nonzero(nan[0])[0]) == {0x7F, 0xFF}
    fin = ~nan
    t = 1e-6 if path == "mma" else TOL[path]
    np.testing.assert_allclose(y[fin], ref[fin], rtol=t, atol=t * np.abs(ref[fin]).max())


@pytest.mark.parametrize("M", [1, 3, 8, 20])
def test_each_position_takes_its_blocks_scale(env, M, path):
    # distinct scales per 16-element block; a one-hot x row k picks element k
    # times its own block's scale (the lanes of a 32-k block hold two blocks)
    K = 512
    nblk = K // 16
    codes = np.full((4, K), 3, np.uint8)  # 1.5 everywhere
    codes[1] = 11                         # -1.5
    sc = ((np.arange(4 * nblk).reshape(4, nblk) % 14 + 1) << 3 | (np.arange(4 * nblk).reshape(4, nblk) % 8))
    sc = sc.astype(np.uint8)
    pos = [0, 7, 8, 15, 16, 23, 24, 31, 32, 255, 256, 300, 511]
    ks = np.array([pos[i % len(pos)] for i in range(M)])
    x = np.zeros((M, K), np.float32)
    x[np.arange(M), ks] = 1.0
    y = _run(env, workloads.f32_to_bf16_bits(x), _pack_codes(codes), sc, 1.0)
    w = oracle.nvfp4_dequant(_pack_codes(codes), sc, 1.0)
    if path == "mma":
        assert np.array_equal(y.astype(np.float64), w[:, ks].T)
    else:
        np.testing.assert_allclose(y, w[:, ks].T, rtol=TOL[path])


@pytest.mark.parametrize("M", [1, 2, 5, 8, 9, 16, 20, 33, 64, 65, 80, 130])
def test_rows_m(env, M, path):
    nib, sc = workloads.nvfp4_weights(300, 1024, seed=M, tensor_id=0)
    x = workloads.bf16_normal(M, 1024, seed=M, tensor_id=1)
    assert _check(env, x, nib, sc, 0.0123) < TOL[path]


@pytest.mark.parametrize("N,K", [(1, 32), (7, 64), (63, 512), (65, 544), (129, 1056), (257, 4096 + 96),
                                 (64, 16384), (33, 8192)])
def test_ragged_shapes(env, N, K, path):
    nib, sc = workloads.nvfp4_weights(N, K, seed=N + K, tensor_id=0, exp_lo=1, exp_hi=14)
    x = workloads.bf16_normal(5, K, seed=N, tensor_id=1)
    assert _check(env, x, nib, sc, 1.0) < TOL[path]


@pytest.mark.parametrize("K,offset", [(544, 1), (1056, 3), (4096 + 96, 8)])
def test_misaligned_scales_are_realigned(env, K, offset, path):
    nib, sc = workloads.nvfp4_weights(70, K, seed=K, tensor_id=0)
    x = workloads.bf16_normal(9, K, seed=K, tensor_id=1)
    assert _check(env, x, nib, sc, 2.0, sc_offset=offset) < TOL[path]


def test_misaligned_scales_rejected_when_in_place(env):
    torch, mxs = env
    nib, sc = workloads.nvfp4_weights(16, 512, seed=1)
    with pytest.raises(mxs.MxsError):
        _run(env, workloads.bf16_normal(2, 512, seed=1), nib, sc, 1.0, sc_offset=4)


@pytest.mark.parametrize("g", [1.0, 2.0 ** -10, 0.37, -1.5, 0.0, 6.0e4])
def test_global_scale(env, g, path):
    nib, sc = workloads.nvfp4_weights(130, 2048, seed=11)
    x = workloads.bf16_normal(6, 2048, seed=11, tensor_id=1)
    y = _run(env, x, nib, sc, g)
    ref = oracle.nvfp4_gemm(x, nib, sc, g)
    if g == 0.0:
        assert np.all(y == 0.0)
    else:
        assert np.all(gemm_row_rel_err(y, ref) < TOL[path])
        # the tensor scale is one multiplication at the end
        y1 = _run(env, x, nib, sc, 1.0)
        np.testing.assert_array_equal(y, (y1 * np.float32(g)).astype(np.float32))


def test_extreme_scales_and_x(env, path):
    # largest finite E4M3 (448) with the largest code, smallest subnormal
    # (2^-9) with the smallest, on x spanning a wide range per row
    K = 256
    rng = np.random.default_rng(6)
    nib, sc = workloads.nvfp4_weights(96, K, seed=6, exp_lo=0, exp_hi=14)
    sc[0] = 0x7E
    sc[1] = 0x01
    sc[2] = 0xFE                           # -448
    nib[0] = 0x77                          # 6.0
    nib[1] = 0x11                          # 0.5
    x = rng.standard_normal((4, K)).astype(np.float32)
    x[1] *= 2.0 ** 60
    x[2] *= 2.0 ** -60
    x[3, ::7] *= 1e4
    assert _check(env, workloads.f32_to_bf16_bits(x), nib, sc, 1.0) < TOL[path]


def test_nonfinite_x_row_gives_nan_row(env, path):
    nib, sc = workloads.nvfp4_weights(40, 256, seed=8)
    x = workloads.bf16_normal(3, 256, seed=8, tensor_id=1)
    x[1, 5] = 0x7FC0  # NaN
    y = _run(env, x, nib, sc, 1.0)
    assert np.all(np.isnan(y[1])) and np.all(np.isfinite(y[[0, 2]]))
    ref = oracle.nvfp4_gemm(x[[0, 2]], nib, sc, 1.0)
    assert np.all(gemm_row_rel_err(y[[0, 2]], ref) < TOL[path])


def test_repeat_calls_identical(env):
    nib, sc = workloads.nvfp4_weights(64, 16384, seed=9)   # split-K path
    x = workloads.bf16_normal(4, 16384, seed=9, tensor_id=1)
    a = _run(env, x, nib, sc, 0.5)
    b = _run(env, x, nib, sc, 0.5)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("M", [5, 20, 64])
def test_lm_head_shape_sampled(env, M, path):
    """The lm_head of an 8B target (K = 4096, N = 128256) with NVFP4 weights,
    in the launch configuration the benchmark times; sampled output columns
    against the oracle."""
    torch, mxs = env
    dev = torch.device("cuda:0")
    N, K = 128256, 4096
    nib, sc = workloads.device_nvfp4_weights(N, K, seed=M, device=dev)
    x = workloads.device_bf16_normal(M, K, seed=M + 1, device=dev)
    g = 0.0731
    y = mxs.nvfp4_verify_gemm(x, nib, sc, g)
    torch.cuda.synchronize()
    cols = np.unique(np.concatenate([np.arange(0, 128), np.arange(N - 130, N),
                                     np.random.default_rng(M).integers(0, N, 512)]))
    tc = torch.from_numpy(cols).to(dev)
    x_bits = x.view(torch.int16).cpu().numpy().view(np.uint16)
    ref = oracle.nvfp4_gemm(x_bits, nib[tc].cpu().numpy(), sc[tc].cpu().numpy(), g)
    got = y[:, tc].cpu().numpy()
    assert np.all(gemm_row_rel_err(got, ref) < TOL[path])
