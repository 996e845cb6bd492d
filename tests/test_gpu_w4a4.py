"""GPU parity of the W4A4 verify GEMM (mxfp4_verify_gemm_w4a4) with the oracle.

"Module 11. Speculative Decoding and Quantization", §12: W4A4 puts the
activations in MX-FP4 too.  The kernel quantises X by the pack rule, 32
elements per block, and runs the block-scaled tensor-core product
(kind::mxf4, one term, passes of up to 256 rows); the oracle quantises X by
the same rule in double and forms the plain product.  Every product of two
E2M1 values and two power-of-two scales is exact in fp32, so what remains is
fp32 summation error: the bar is 1e-5 of each row's largest |Y|.
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import bf16_tensor_from_bits, cuda_or_skip, gemm_row_rel_err

pytestmark = pytest.mark.gpu

W4A4_REL_TOL = 1e-5


@pytest.fixture
def env():
    return cuda_or_skip()


def _dev(env, x, nib, sc):
    torch, _ = env
    dev = torch.device("cuda:0")
    return bf16_tensor_from_bits(torch, x, dev), torch.from_numpy(nib).to(dev), torch.from_numpy(sc).to(dev)


def _run(env, x, nib, sc, **kw):
    torch, mxs = env
    y = mxs.mxfp4_verify_gemm_w4a4(*_dev(env, x, nib, sc), **kw)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def _check(env, x, nib, sc, cols=None):
    y = _run(env, x, nib, sc)
    if cols is not None:
        y = y[:, cols]
        nib, sc = nib[cols], sc[cols]
    ref = oracle.gemm_w4a4(x, nib, sc)
    err = gemm_row_rel_err(y, ref)
    assert np.all(err <= W4A4_REL_TOL), f"max rel err {err.max():.3e} (row {int(err.argmax())})"
    return y, ref


@pytest.mark.parametrize("M", [1, 5, 16, 17, 31, 64, 80, 100, 128, 129, 192, 193, 200, 240, 256, 257, 300, 520])
def test_w4a4_rows_m(env, M):
    nib, sc = workloads.mxfp4_weights(300, 1024, 118, 132, seed=M, tensor_id=0)
    x = workloads.bf16_normal(M, 1024, seed=M, tensor_id=1)
    _check(env, x, nib, sc)


@pytest.mark.parametrize("M", [80, 200])
@pytest.mark.parametrize("N,K", [(1, 32), (7, 64), (1, 128), (127, 512), (65, 544), (129, 640), (200, 4096),
                                 (257, 2176), (1000, 14336), (130, 8192 + 32), (64, 384), (33, 96)])
def test_w4a4_ragged(env, M, N, K):
    nib, sc = workloads.mxfp4_weights(N, K, 118, 132, seed=N + K, tensor_id=0)
    x = workloads.bf16_normal(M, K, seed=N + K, tensor_id=1)
    _check(env, x, nib, sc)


def test_w4a4_every_weight_code(env):
    K = 128
    codes = np.arange(16, dtype=np.uint8).repeat(K).reshape(16, K)
    nib = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sc = np.full((16, K // 32), 127, dtype=np.uint8)
    x = workloads.bf16_normal(100, K, seed=1)
    _check(env, x, nib, sc)


def test_w4a4_rounding_cases_exact(env):
    # blocks whose only nonzero element is a tie or a scale boundary of the
    # rule (5 -> 4, 7 -> 8, 13 -> 12, 2.5 -> 2, ...), weights all 1.0: the
    # output is the quantised value itself, bit for bit
    vals = np.array([5.0, -5.0, 7.0, 13.0, 2.5, 0.25, 6.0, 0.75, 3.5, -3.5, 1.25, 24.0, 28.0, 0.1, 1e-3, 96.0],
                    dtype=np.float32)
    K = 64
    x = np.zeros((len(vals), K), dtype=np.float32)
    x[:, 7] = vals
    nib = np.full((130, K // 2), 0x22, dtype=np.uint8)
    sc = np.full((130, K // 32), 127, dtype=np.uint8)
    xb = workloads.f32_to_bf16_bits(x)
    y = _run(env, xb, nib, sc)
    assert np.array_equal(y, oracle.gemm_w4a4(xb, nib, sc).astype(np.float32))


def test_w4a4_nan_scale_and_nonfinite_rows(env):
    K = 256
    nib, sc = workloads.mxfp4_weights(200, K, 118, 132, seed=6, tensor_id=0)
    sc[3, 2] = 255
    x = workloads.bf16_normal(90, K, seed=6)
    x[10, 100] = 0x7F80  # +inf
    x[40, 3] = 0xFFC0    # NaN
    y = _run(env, x, nib, sc)
    ref = oracle.gemm_w4a4(x, nib, sc)
    assert np.all(np.isnan(y[:, 3])) and np.all(np.isnan(y[10])) and np.all(np.isnan(y[40]))
    ok_r = np.setdiff1d(np.arange(90), [10, 40])
    ok_c = np.setdiff1d(np.arange(200), [3])
    yy, rr = y[np.ix_(ok_r, ok_c)], ref[np.ix_(ok_r, ok_c)]
    assert np.all(np.isfinite(yy))
    assert np.all(gemm_row_rel_err(yy, rr) <= W4A4_REL_TOL)


@pytest.mark.parametrize("scale", [2.0 ** -131, 2.0 ** -127, 2.0 ** -120, 1e-3, 3e4, 2.0 ** 100])
def test_w4a4_activation_magnitudes(env, scale):
    # rows far below 1 (down to bf16 subnormals, where the rule's clamp of
    # the block exponent at -127 rounds most elements to 0) and far above
    nib, sc = workloads.mxfp4_weights(160, 512, 118, 132, seed=9)
    rng = np.random.default_rng(9)
    xf = (rng.standard_normal((96, 512)) * scale).astype(np.float32)
    xf[1] *= 1e-3
    _check(env, workloads.f32_to_bf16_bits(xf), nib, sc)


def test_w4a4_zero_rows_and_blocks(env):
    K = 512
    nib, sc = workloads.mxfp4_weights(140, K, 118, 132, seed=4)
    x = workloads.bf16_normal(84, K, seed=4)
    x[0] = 0
    x[5, 64:256] = 0
    x[7, ::2] = 0x8000  # negative zeros
    y, _ = _check(env, x, nib, sc)
    assert np.all(y[0] == 0)


def test_w4a4_wide_spread_within_block(env):
    # a block maximum far above its neighbours: the neighbours quantise to 0
    # or to the block's coarse grid, exactly as the rule says
    K = 512
    rng = np.random.default_rng(2)
    xf = rng.standard_normal((120, K)).astype(np.float32)
    xf[:, ::32] *= 2.0 ** 12
    xf[:, 5::32] *= 2.0 ** -20
    nib, sc = workloads.mxfp4_weights(96, K, 118, 132, seed=2)
    _check(env, workloads.f32_to_bf16_bits(xf), nib, sc)


def test_w4a4_split_k_and_deterministic(env):
    torch, mxs = env
    nib, sc = workloads.mxfp4_weights(1000, 14336, 118, 132, seed=4)
    xb = workloads.bf16_normal(200, 14336, seed=4)
    x, nd, sd = _dev(env, xb, nib, sc)
    status = torch.zeros(1, dtype=torch.int32, device=x.device)
    a = mxs.mxfp4_verify_gemm_w4a4(x, nd, sd, dev_status=status)
    b = mxs.mxfp4_verify_gemm_w4a4(x, nd, sd)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    err = gemm_row_rel_err(a.cpu().numpy(), oracle.gemm_w4a4(xb, nib, sc))
    assert np.all(err <= W4A4_REL_TOL)


@pytest.mark.parametrize("splits", ["1", "3", "7"])
def test_w4a4_forced_splits(env, monkeypatch, splits):
    monkeypatch.setenv("MXS_GEMM_SPLITS", splits)
    nib, sc = workloads.mxfp4_weights(300, 4096, 118, 132, seed=7)
    x = workloads.bf16_normal(150, 4096, seed=7)
    _check(env, x, nib, sc)


def test_w4a4_caller_workspace_and_output(env):
    torch, mxs = env
    nib, sc = workloads.mxfp4_weights(500, 2048, 118, 132, seed=8)
    xb = workloads.bf16_normal(230, 2048, seed=8)
    x, nd, sd = _dev(env, xb, nib, sc)
    ws = torch.empty(mxs.mxfp4_verify_gemm_w4a4_workspace_size(230, 500, 2048), dtype=torch.uint8, device=x.device)
    out = torch.full((230, 500), float("nan"), dtype=torch.float32, device=x.device)
    y = mxs.mxfp4_verify_gemm_w4a4(x, nd, sd, out=out, workspace=ws)
    torch.cuda.synchronize()
    assert y.data_ptr() == out.data_ptr()
    err = gemm_row_rel_err(out.cpu().numpy(), oracle.gemm_w4a4(xb, nib, sc))
    assert np.all(err <= W4A4_REL_TOL)


@pytest.mark.parametrize("idx,name,K,N", [(i,) + s for i, s in
                                           enumerate(list(workloads.LLAMA8B_LAYER) + [workloads.LLAMA8B_LM_HEAD])])
@pytest.mark.parametrize("M", [80, 256])
def test_w4a4_llama8b_shapes_sampled(env, idx, name, K, N, M):
    # the full weight shapes, in the launch configuration of the benchmark;
    # the oracle checks 384 sampled output columns (and the last one)
    nib, sc = workloads.mxfp4_weights(N, K, *workloads.LLAMA_EXP_RANGE, seed=0, tensor_id=200 + idx)
    x = workloads.bf16_normal(M, K, seed=0, tensor_id=8)
    rng = np.random.default_rng(idx)
    cols = np.unique(np.concatenate([rng.choice(N, size=min(N, 384), replace=False), [N - 1]]))
    _check(env, x, nib, sc, cols=cols)


@pytest.mark.parametrize("M", [80, 300])
def test_w4a4_grouped_equals_single_without_split(env, monkeypatch, M):
    # the grouped form never splits K; with splitting off, each problem's
    # single call runs the same kernel on the same quantised X: the same bits
    torch, mxs = env
    dev = torch.device("cuda:0")
    monkeypatch.setenv("MXS_GEMM_SPLITS", "1")
    probs = []
    xs = {K: bf16_tensor_from_bits(torch, workloads.bf16_normal(M, K, seed=K, tensor_id=M), dev) for K in (4096, 14336)}
    for i, (K, N) in enumerate([(4096, 6144), (14336, 4096), (4096, 1000), (4096, 6144)]):
        nib, sc = workloads.mxfp4_weights(N, K, 118, 132, seed=i, tensor_id=400 + i)
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
        probs.append((xs[K], torch.from_numpy(nib).to(dev), torch.from_numpy(sc).to(dev), y))
    mxs.mxfp4_verify_gemm_grouped(probs, w4a4=True)
    for x, nib, sc, y in probs:
        single = mxs.mxfp4_verify_gemm_w4a4(x, nib, sc)
        torch.cuda.synchronize()
        assert torch.equal(single.view(torch.int32), y.view(torch.int32))


def test_w4a4_grouped_plan_against_oracle(env):
    torch, mxs = env
    dev = torch.device("cuda:0")
    M = 130
    xb = {K: workloads.bf16_normal(M, K, seed=3, tensor_id=K) for K in (512, 1024)}
    xd = {K: bf16_tensor_from_bits(torch, v, dev) for K, v in xb.items()}
    host, probs = [], []
    for i, (K, N) in enumerate([(1024, 300), (512, 129), (1024, 77)]):
        nib, sc = workloads.mxfp4_weights(N, K, 118, 132, seed=i, tensor_id=500 + i)
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
        host.append((K, nib, sc))
        probs.append((xd[K], torch.from_numpy(nib).to(dev), torch.from_numpy(sc).to(dev), y))
    plan = mxs.GroupedGemm(probs, w4a4=True)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    plan(dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for (K, nib, sc), (_, _, _, y) in zip(host, probs):
        err = gemm_row_rel_err(y.cpu().numpy(), oracle.gemm_w4a4(xb[K], nib, sc))
        assert np.all(err <= W4A4_REL_TOL)
