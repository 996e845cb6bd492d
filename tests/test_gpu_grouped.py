"""GPU parity of mxfp4_verify_gemm_grouped (many independent GEMMs per call)
against the CPU oracle, and against the single-GEMM entry point."""
import numpy as np
import pytest

import oracle
import workloads
from helpers import GEMM_REL_TOL, bf16_tensor_from_bits, cuda_or_skip, gemm_row_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    return cuda_or_skip()


def _problems(env, M, shapes, n_x=2, seed=0):
    torch, mxs = env
    dev = torch.device("cuda:0")
    xs = {}
    host = []
    probs = []
    for i, (K, N) in enumerate(shapes):
        key = (K, i % n_x)
        if key not in xs:
            bits = workloads.bf16_normal(M, K, seed=seed + len(xs), tensor_id=K)
            xs[key] = (bits, bf16_tensor_from_bits(torch, bits, dev))
        nib, sc = workloads.mxfp4_weights(N, K, 118, 132, seed=seed, tensor_id=100 + i)
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
        probs.append((xs[key][1], torch.from_numpy(nib).to(dev), torch.from_numpy(sc).to(dev), y))
        host.append((xs[key][0], nib, sc))
    return probs, host


@pytest.mark.parametrize("M", [1, 5, 20, 64, 80, 130])
def test_grouped_matches_oracle(env, M):
    torch, mxs = env
    shapes = [(512, 100), (4096, 640), (1024, 64), (512, 1), (2048, 257), (4096, 1000)]
    probs, host = _problems(env, M, shapes)
    mxs.mxfp4_verify_gemm_grouped(probs)
    torch.cuda.synchronize()
    for (x, nib, sc), (_, _, _, y) in zip(host, probs):
        err = gemm_row_rel_err(y.cpu().numpy(), oracle.gemm(x, nib, sc))
        assert np.all(err <= GEMM_REL_TOL), f"max rel err {err.max():.3e}"


def test_grouped_llama8b_layer_and_head(env):
    torch, mxs = env
    shapes = [(K, N) for _, K, N in workloads.LLAMA8B_LAYER] + [workloads.LLAMA8B_LM_HEAD[1:]]
    probs, host = _problems(env, 5, shapes, n_x=1)
    mxs.mxfp4_verify_gemm_grouped(probs)
    torch.cuda.synchronize()
    for (x, nib, sc), (_, _, _, y) in zip(host, probs):
        err = gemm_row_rel_err(y.cpu().numpy(), oracle.gemm(x, nib, sc))
        assert np.all(err <= GEMM_REL_TOL), f"max rel err {err.max():.3e}"


def test_grouped_many_problems_several_launches(env):
    torch, mxs = env
    shapes = [(512 * (1 + i % 3), 64 + 7 * i) for i in range(150)]
    probs, host = _problems(env, 5, shapes, n_x=3)
    mxs.mxfp4_verify_gemm_grouped(probs)
    torch.cuda.synchronize()
    for (x, nib, sc), (_, _, _, y) in zip(host, probs):
        err = gemm_row_rel_err(y.cpu().numpy(), oracle.gemm(x, nib, sc))
        assert np.all(err <= GEMM_REL_TOL)


def test_grouped_equals_single_call_without_split(env, monkeypatch):
    torch, mxs = env
    # with K unsplit in the single call, the two paths add in the same order
    monkeypatch.setenv("MXS_GEMM_SPLITS", "1")
    probs, host = _problems(env, 5, [(4096, 28672), (4096, 6144)], n_x=1)
    mxs.mxfp4_verify_gemm_grouped(probs)
    for x, nib, sc, y in probs:
        single = mxs.mxfp4_verify_gemm(x, nib, sc)
        torch.cuda.synchronize()
        assert torch.equal(single.view(torch.int32), y.view(torch.int32))


def test_grouped_equals_single_call_tcgen05(env, monkeypatch):
    torch, mxs = env
    # both entry points on the tcgen05 kernel (K is never split there)
    monkeypatch.setenv("MXS_GEMM_PATH", "umma")
    probs, host = _problems(env, 40, [(4096, 28672), (14336, 4096)], n_x=1)
    mxs.mxfp4_verify_gemm_grouped(probs)
    for x, nib, sc, y in probs:
        single = mxs.mxfp4_verify_gemm(x, nib, sc)
        torch.cuda.synchronize()
        assert torch.equal(single.view(torch.int32), y.view(torch.int32))


def test_grouped_many_problems_several_launches_wide(env):
    torch, mxs = env
    shapes = [(512 * (1 + i % 3), 64 + 7 * i) for i in range(150)]
    probs, host = _problems(env, 40, shapes, n_x=3)
    mxs.mxfp4_verify_gemm_grouped(probs)
    torch.cuda.synchronize()
    for (x, nib, sc), (_, _, _, y) in zip(host, probs):
        err = gemm_row_rel_err(y.cpu().numpy(), oracle.gemm(x, nib, sc))
        assert np.all(err <= GEMM_REL_TOL)


def test_grouped_rejects_unsupported(env):
    torch, mxs = env
    probs, _ = _problems(env, 5, [(544, 64)])
    with pytest.raises(mxs.MxsError):
        mxs.mxfp4_verify_gemm_grouped(probs)


@pytest.mark.parametrize("M", [5, 20])
def test_grouped_claim_order_does_not_change_results(env, monkeypatch, M):
    torch, mxs = env
    # items claimed from the counter (longest first) vs the static round robin:
    # every output element is computed by one item in a fixed order either way
    shapes = [(K, N) for _, K, N in workloads.LLAMA8B_LAYER] * 3 + [(512, 300), (14336, 70)]
    probs, _ = _problems(env, M, shapes, n_x=1)
    mxs.mxfp4_verify_gemm_grouped(probs)
    torch.cuda.synchronize()
    dyn = [y.clone() for *_, y in probs]
    monkeypatch.setenv("MXS_GEMM_SCHED", "static")
    for *_, y in probs:
        y.fill_(float("nan"))
    mxs.mxfp4_verify_gemm_grouped(probs)
    torch.cuda.synchronize()
    for a, (*_, b) in zip(dyn, probs):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("M", [5, 20])
def test_grouped_plan_equals_the_call(env, M):
    """GroupedGemm (checked once, one C call per step) writes the same bits as
    mxfp4_verify_gemm_grouped, call after call, and sees in-place updates of x."""
    torch, mxs = env
    shapes = [(4096, 640), (1024, 64), (2048, 257), (4096, 1000)]
    probs, _ = _problems(env, M, shapes)
    mxs.mxfp4_verify_gemm_grouped(probs)
    torch.cuda.synchronize()
    ref = [p[3].clone() for p in probs]
    plan = mxs.GroupedGemm(probs)
    for _ in range(3):
        for p in probs:
            p[3].fill_(float("nan"))
        plan()
        torch.cuda.synchronize()
        for p, r in zip(probs, ref):
            assert torch.equal(p[3].view(torch.int32), r.view(torch.int32))
    x0 = probs[0][0]
    x0.mul_(2.0)  # exact: a power of two
    plan()
    torch.cuda.synchronize()
    assert torch.equal(probs[0][3], 2.0 * ref[0])
