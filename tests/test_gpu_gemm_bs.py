"""GPU parity of the block-scaled tensor-core verify GEMM, both kinds:
kind::mxf8f6f4 (X as two E4M3 terms) and kind::mxf4 (X as six E2M1 terms).

The entry points take this path for passes of 9 or more rows (mxf4 up to 32
rows, mxf8f6f4 beyond); here each kind is forced (MXS_GEMM_PATH=bs8 / bs4)
so that narrow, ragged and pathological shapes exercise both, against the
same oracle and bar as every other path.
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import GEMM_REL_TOL, bf16_tensor_from_bits, cuda_or_skip, gemm_row_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["bs8", "bs4"])
def env(request, monkeypatch):
    monkeypatch.setenv("MXS_GEMM_PATH", request.param)
    return cuda_or_skip()


def _run(env, x, nib, sc, **kw):
    torch, mxs = env
    dev = torch.device("cuda:0")
    y = mxs.mxfp4_verify_gemm(bf16_tensor_from_bits(torch, x, dev), torch.from_numpy(nib).to(dev),
                              torch.from_numpy(sc).to(dev), **kw)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def _check(env, x, nib, sc):
    y = _run(env, x, nib, sc)
    ref = oracle.gemm(x, nib, sc)
    err = gemm_row_rel_err(y, ref)
    assert np.all(err <= GEMM_REL_TOL), f"max rel err {err.max():.3e}"
    return y, ref


@pytest.mark.parametrize("M", [1, 5, 9, 16, 17, 20, 32, 33, 48, 63, 64, 65, 80, 96, 112, 128, 129, 200])
def test_bs_rows_m(env, M):
    nib, sc = workloads.mxfp4_weights(300, 1024, 118, 132, seed=M, tensor_id=0)
    x = workloads.bf16_normal(M, 1024, seed=M, tensor_id=1)
    y, ref = _check(env, x, nib, sc)
    # two E4M3 terms hold bf16 N(0,1) exactly, six E2M1 terms to ~1e-7 of
    # each block maximum: what remains is fp32 summation error
    assert np.all(gemm_row_rel_err(y, ref) < 1e-5)


@pytest.mark.parametrize("N,K", [(1, 32), (7, 64), (1, 128), (127, 512), (65, 544), (129, 640), (200, 4096),
                                 (257, 2176), (1000, 14336), (130, 8192 + 32), (64, 384), (33, 96)])
def test_bs_ragged(env, N, K):
    nib, sc = workloads.mxfp4_weights(N, K, 118, 132, seed=N + K, tensor_id=0)
    x = workloads.bf16_normal(20, K, seed=N + K, tensor_id=1)
    _check(env, x, nib, sc)


def test_bs_every_code(env):
    K = 128
    codes = np.arange(16, dtype=np.uint8).repeat(K).reshape(16, K)
    nib = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sc = np.full((16, K // 32), 127, dtype=np.uint8)
    x = workloads.bf16_normal(12, K, seed=1)
    y, ref = _check(env, x, nib, sc)
    assert np.all(gemm_row_rel_err(y, ref) < 1e-6)


def test_bs_every_weight_exponent(env):
    # E8M0 bytes 0..230 straight into the tensor core's factors, one block each
    # (larger exponents overflow fp32 outputs in the oracle's terms as well)
    E = 231
    K = 32 * E
    rng = np.random.default_rng(5)
    nib = rng.integers(0, 256, size=(E, K // 2), dtype=np.uint8)
    sc = np.full((E, K // 32), 127, dtype=np.uint8)
    for n in range(E):
        sc[n, n] = n  # row n: block n carries exponent n, the rest 2^0
    K128 = (K + 127) // 128 * 128
    nib = np.pad(nib, ((0, 0), (0, (K128 - K) // 2)))
    sc = np.pad(sc, ((0, 0), (0, (K128 - K) // 32)), constant_values=127)
    x = workloads.bf16_normal(20, K128, seed=5)
    _check(env, x, nib, sc)


@pytest.mark.parametrize("lo,hi", [(0, 200), (100, 140), (60, 61)])
def test_bs_exponent_spreads(env, lo, hi):
    rng = np.random.default_rng(lo)
    N, K = 256, 1024
    nib = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sc = rng.integers(lo, hi + 1, size=(N, K // 32)).astype(np.uint8)
    sc[0, :] = lo
    x = workloads.bf16_normal(20, K, seed=lo)
    _check(env, x, nib, sc)


def test_bs_isolated_small_blocks(env):
    N, K = 128, 512
    codes = np.full((N, K), 7, dtype=np.uint8)  # 6.0
    nib = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sc = np.full((N, K // 32), 160, dtype=np.uint8)
    sc[5, 3] = 100
    sc[6, :] = 100
    sc[6, 9] = 130
    x = workloads.bf16_normal(16, K, seed=3)
    _check(env, x, nib, sc)


def test_bs_nan_scale(env):
    K = 128
    nib = np.full((3, K // 2), 0x22, dtype=np.uint8)
    sc = np.full((3, K // 32), 127, dtype=np.uint8)
    sc[0, 2] = 255
    x = workloads.f32_to_bf16_bits(np.ones((12, K), dtype=np.float32))
    y = _run(env, x, nib, sc)
    assert np.all(np.isnan(y[:, 0])) and np.all(y[:, 1:] == 128.0)


@pytest.mark.parametrize("scale", [2.0 ** -120, 1e-3, 3e4, 2.0 ** 100])
def test_bs_activation_magnitudes(env, scale):
    nib, sc = workloads.mxfp4_weights(160, 512, 118, 132, seed=9)
    rng = np.random.default_rng(9)
    xf = (rng.standard_normal((20, 512)) * scale).astype(np.float32)
    xf[1] *= 1e-3
    _check(env, workloads.f32_to_bf16_bits(xf), nib, sc)


def test_bs_activation_spread_within_block(env):
    # elements far below their block's largest: the second E4M3 term and its
    # own scale keep them
    K = 512
    rng = np.random.default_rng(2)
    xf = rng.standard_normal((20, K)).astype(np.float32)
    xf[:, ::32] *= 2.0 ** 12
    xf[:, 5::32] *= 2.0 ** -20
    nib, sc = workloads.mxfp4_weights(96, K, 118, 132, seed=2)
    _check(env, workloads.f32_to_bf16_bits(xf), nib, sc)


def test_bs_split_k_and_deterministic(env):
    torch, mxs = env
    dev = torch.device("cuda:0")
    # 8 tiles of 128 rows: K is split over the idle SMs
    nib, sc = workloads.mxfp4_weights(1000, 14336, 118, 132, seed=4)
    xb = workloads.bf16_normal(40, 14336, seed=4)
    x = bf16_tensor_from_bits(torch, xb, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    nd, sd = torch.from_numpy(nib).to(dev), torch.from_numpy(sc).to(dev)
    a = mxs.mxfp4_verify_gemm(x, nd, sd, dev_status=status)
    b = mxs.mxfp4_verify_gemm(x, nd, sd)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    err = gemm_row_rel_err(a.cpu().numpy(), oracle.gemm(xb, nib, sc))
    assert np.all(err <= GEMM_REL_TOL)


@pytest.mark.parametrize("splits", ["1", "3", "7"])
def test_bs_forced_splits(env, monkeypatch, splits):
    monkeypatch.setenv("MXS_GEMM_SPLITS", splits)
    nib, sc = workloads.mxfp4_weights(300, 4096, 118, 132, seed=7)
    x = workloads.bf16_normal(33, 4096, seed=7)
    _check(env, x, nib, sc)


@pytest.mark.parametrize("idx,name,K,N", [(i,) + s for i, s in
                                           enumerate(list(workloads.LLAMA8B_LAYER) + [workloads.LLAMA8B_LM_HEAD])])
@pytest.mark.parametrize("M", [20, 64])
def test_bs_llama8b_layer(env, idx, name, K, N, M):
    nib, sc = workloads.mxfp4_weights(N, K, *workloads.LLAMA_EXP_RANGE, seed=0, tensor_id=200 + idx)
    x = workloads.bf16_normal(M, K, seed=0, tensor_id=8)
    _check(env, x, nib, sc)


def test_bs_grouped_equals_single_without_split(env, monkeypatch):
    torch, mxs = env
    dev = torch.device("cuda:0")
    monkeypatch.setenv("MXS_GEMM_SPLITS", "1")
    probs = []
    for i, (K, N) in enumerate([(4096, 6144), (14336, 4096), (4096, 1000)]):
        nib, sc = workloads.mxfp4_weights(N, K, 118, 132, seed=i, tensor_id=300 + i)
        x = bf16_tensor_from_bits(torch, workloads.bf16_normal(48, K, seed=i, tensor_id=K), dev)
        y = torch.full((48, N), float("nan"), dtype=torch.float32, device=dev)
        probs.append((x, torch.from_numpy(nib).to(dev), torch.from_numpy(sc).to(dev), y))
    mxs.mxfp4_verify_gemm_grouped(probs)
    for x, nib, sc, y in probs:
        single = mxs.mxfp4_verify_gemm(x, nib, sc)
        torch.cuda.synchronize()
        assert torch.equal(single.view(torch.int32), y.view(torch.int32))
