"""GPU parity of mxfp4_pack against the CPU oracle: bit-exact nibbles and
scales (integer / byte output)."""
import numpy as np
import pytest

import oracle
import workloads
from helpers import cuda_or_skip

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    return cuda_or_skip()


def _gpu_pack(env, w, dtype):
    torch, mxs = env
    dev = torch.device("cuda:0")
    if dtype == "f32":
        t = torch.from_numpy(np.ascontiguousarray(w, np.float32)).to(dev)
    else:
        t = torch.from_numpy(np.ascontiguousarray(w).view(np.int16)).to(dev).view(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    nib, sc = mxs.mxfp4_pack(t, dev_status=status)
    torch.cuda.synchronize()
    return nib.cpu().numpy(), sc.cpu().numpy(), int(status.item())


def _weights(kind, N, K, seed):
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((N, K)).astype(np.float32)
    if kind == "scaled":
        w *= (10.0 ** rng.uniform(-30, 30, size=(N, 1))).astype(np.float32)
    elif kind == "ties":
        grid = np.array([0, 0.25, 0.5, 0.75, 1, 1.25, 1.5, 1.75, 2, 2.5, 3, 3.5, 4, 5, 6], np.float32)
        w = rng.choice(grid, size=(N, K)) * np.where(rng.random((N, K)) < 0.5, -1, 1).astype(np.float32)
        w[:, ::32] = 6.0
        w *= np.float32(2.0) ** rng.integers(-20, 20, size=(N, 1)).astype(np.float32)
    elif kind == "sparse":
        w[rng.random((N, K)) < 0.7] = 0.0
        w[:, :32] = 0.0
        w[:, K // 2 + 3] = -0.0
    elif kind == "tiny":
        w = (w * np.float32(1e-39)).astype(np.float32)  # subnormal fp32 inputs
    return w


@pytest.mark.parametrize("kind", ["normal", "scaled", "ties", "sparse", "tiny"])
@pytest.mark.parametrize("N,K", [(1, 32), (33, 96), (256, 512), (300, 4096)])
def test_pack_f32_bit_exact(env, kind, N, K):
    w = _weights(kind, N, K, N + K)
    nib, sc, status = _gpu_pack(env, w, "f32")
    rn, rs, ok = oracle.pack(w)
    assert ok and status == 0
    assert np.array_equal(sc, rs) and np.array_equal(nib, rn)


@pytest.mark.parametrize("kind", ["normal", "scaled", "ties", "sparse"])
def test_pack_bf16_bit_exact(env, kind):
    w = _weights(kind, 64, 1024, 3)
    bits = workloads.f32_to_bf16_bits(w)
    nib, sc, status = _gpu_pack(env, bits, "bf16")
    rn, rs, ok = oracle.pack(bits, dtype="bf16")
    assert np.array_equal(sc, rs) and np.array_equal(nib, rn)


def test_pack_nonfinite_flagged(env):
    w = _weights("normal", 4, 128, 1)
    w[1, 5] = np.inf
    w[2, 70] = np.nan
    nib, sc, status = _gpu_pack(env, w, "f32")
    rn, rs, ok = oracle.pack(w)
    assert not ok and status & 0x20
    assert np.array_equal(sc, rs) and np.array_equal(nib, rn)


def test_pack_then_gemm_roundtrip(env):
    torch, mxs = env
    dev = torch.device("cuda:0")
    w = _weights("normal", 512, 2048, 11)
    nib, sc, _ = _gpu_pack(env, w, "f32")
    x = workloads.bf16_normal(5, 2048, seed=11)
    ref = oracle.gemm(x, nib, sc)
    from helpers import bf16_tensor_from_bits, gemm_row_rel_err
    y = mxs.mxfp4_verify_gemm(bf16_tensor_from_bits(torch, x, dev), torch.from_numpy(nib).to(dev),
                              torch.from_numpy(sc).to(dev))
    torch.cuda.synchronize()
    assert np.all(gemm_row_rel_err(y.cpu().numpy(), ref) <= 2e-3)
