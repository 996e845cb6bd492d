"""GPU parity of the MX-FP4 KV cache of the verification block
(``mxfp4_kv_append``, ``spec_kv_commit``, ``mxfp4_kv_dequant``) against the
oracle, bit for bit ("Next-Gen Speculative Decoding and FP4 Quantization ...":
the FP4 KV cache pool; "Module 11. Speculative Decoding and Quantization" §4:
the unaccepted suffix and its cache entries are discarded).

The quantisation, the placement at the committed length, the untouched
positions, the commit arithmetic and the decoded values are all integer or
exact, so every comparison is exact (NaN compared as NaN).
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import cuda_or_skip

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    return cuda_or_skip()


def _kv_rows(B, T, W, seed):
    """K/V-like rows: N(0, 1) with a per-head (128-wide) magnitude from 2^-6 to 2^6."""
    rng = workloads.host_rng(seed, 60)
    x = rng.standard_normal((B, T, W), dtype=np.float32)
    heads = max(1, W // 128)
    mag = np.exp2(rng.integers(-6, 7, size=(B, T, heads))).astype(np.float32)
    return (x * np.repeat(mag, W // heads, axis=2)[:, :, :W]).astype(np.float32)


def _cache(B, L, W, seed):
    rng = workloads.host_rng(seed, 61)
    return (rng.integers(0, 256, size=(B, L, W // 2), dtype=np.uint8),
            rng.integers(0, 256, size=(B, L, W // 32), dtype=np.uint8))


def _to(torch, a, dev):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def _append_gpu(env, kv, nib, sc, lens, dtype):
    torch, mxs = env
    dev = torch.device("cuda:0")
    t_kv = _to(torch, kv, dev)
    if dtype == "bf16":
        t_kv = _to(torch, kv.view(np.int16), dev).view(torch.bfloat16)
    t_nib, t_sc, t_len = _to(torch, nib, dev), _to(torch, sc, dev), _to(torch, lens, dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    mxs.mxfp4_kv_append(t_kv, t_nib, t_sc, t_len, dev_status=st)
    torch.cuda.synchronize()
    return t_nib.cpu().numpy(), t_sc.cpu().numpy(), int(st.item())


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,T,L,W", [(1, 5, 16, 32), (4, 5, 64, 1024), (3, 8, 40, 4128), (64, 5, 512, 1024),
                                     (2, 1, 3, 64), (5, 33, 40, 256)])
def test_append_bit_exact(env, dtype, B, T, L, W):
    kv = _kv_rows(B, T, W, seed=B * T + W)
    if dtype == "bf16":
        kv = workloads.f32_to_bf16_bits(kv)
    nib, sc = _cache(B, L, W, seed=L)
    lens = workloads.host_rng(W, 62).integers(0, L - T + 1, size=B).astype(np.int32)
    g_nib, g_sc, st = _append_gpu(env, kv, nib.copy(), sc.copy(), lens, dtype)
    full = oracle.kv_append(kv, nib, sc, lens, dtype=dtype)
    assert full == 0 and st == 0
    assert np.array_equal(g_nib, nib) and np.array_equal(g_sc, sc)


def test_append_past_the_end_flags_and_skips(env):
    torch, mxs = env
    B, T, L, W = 6, 5, 20, 256
    kv = _kv_rows(B, T, W, seed=9)
    nib, sc = _cache(B, L, W, seed=9)
    lens = np.array([15, 16, 18, 19, 20, 40], np.int32)
    g_nib, g_sc, st = _append_gpu(env, kv, nib.copy(), sc.copy(), lens, "f32")
    full = oracle.kv_append(kv, nib, sc, lens)
    assert full == 0 + 1 + 3 + 4 + 5 + 5
    assert st & mxs.DEV_FLAGS["KV_FULL"]
    assert np.array_equal(g_nib, nib) and np.array_equal(g_sc, sc)


def test_nonfinite_blocks(env):
    torch, mxs = env
    B, T, L, W = 2, 3, 8, 128
    kv = _kv_rows(B, T, W, seed=11)
    kv[0, 1, 5] = np.nan
    kv[1, 2, 100] = np.inf
    nib, sc = _cache(B, L, W, seed=11)
    lens = np.array([0, 4], np.int32)
    g_nib, g_sc, st = _append_gpu(env, kv, nib.copy(), sc.copy(), lens, "f32")
    oracle.kv_append(kv, nib, sc, lens)
    assert st & mxs.DEV_FLAGS["NONFINITE"]
    assert np.array_equal(g_nib, nib) and np.array_equal(g_sc, sc)
    assert g_sc[0, 1, 0] == 255 and g_sc[1, 6, 3] == 255


def test_commit_matches_oracle(env):
    torch, mxs = env
    dev = torch.device("cuda:0")
    rng = workloads.host_rng(12, 63)
    L = 300
    lens = rng.integers(0, L + 1, size=1000).astype(np.int32)
    n = rng.integers(-1, 9, size=1000).astype(np.int32)
    t_len = _to(torch, lens, dev)
    mxs.spec_kv_commit(t_len, _to(torch, n, dev), L)
    torch.cuda.synchronize()
    assert np.array_equal(t_len.cpu().numpy(), oracle.kv_commit(lens, n, L))


@pytest.mark.parametrize("B,L,W", [(1, 8, 32), (4, 33, 1024), (3, 17, 4128)])
def test_dequant_bit_exact(env, B, L, W):
    torch, mxs = env
    dev = torch.device("cuda:0")
    nib, sc = _cache(B, L, W, seed=B + L)  # every code and every scale byte, 255 (NaN) and 254 included
    sc.reshape(-1)[:256] = np.arange(256, dtype=np.uint8)[: min(256, sc.size)]
    lens = workloads.host_rng(W, 64).integers(0, L + 1, size=B).astype(np.int32)
    out = mxs.mxfp4_kv_dequant(_to(torch, nib, dev), _to(torch, sc, dev), _to(torch, lens, dev))
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    ref = oracle.kv_dequant(nib, sc, lens).astype(np.float32)  # exact in fp32, or its overflow to inf
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def test_a_verification_cycle(env):
    """Append a prompt, then one verification block per sequence; acceptance
    (spec_accept on the GPU, the oracle's acceptance on the host, counts
    bit-exact) decides what is kept; commit; read back."""
    torch, mxs = env
    dev = torch.device("cuda:0")
    B, K, V, L, W = 16, 4, 1024, 64, 512
    T = K + 1
    nib, sc = _cache(B, L, W, seed=20)
    nib[:] = 0
    sc[:] = 0
    lens0 = workloads.host_rng(21, 65).integers(1, 30, size=B).astype(np.int32)
    prompt = _kv_rows(B, 30, W, seed=22)
    block = _kv_rows(B, T, W, seed=23)
    p, q, d, u = workloads.spec_inputs(B, K, V, seed=24, logit_std=3.0, draft_noise=0.4)

    # GPU chain
    t_nib, t_sc = _to(torch, nib, dev), _to(torch, sc, dev)
    t_len = torch.zeros(B, dtype=torch.int32, device=dev)
    mxs.mxfp4_kv_append(_to(torch, prompt, dev), t_nib, t_sc, t_len)
    mxs.spec_kv_commit(t_len, _to(torch, lens0, dev), L)  # the prompts' lengths
    mxs.mxfp4_kv_append(_to(torch, block, dev), t_nib, t_sc, t_len)
    _, n_emit = mxs.spec_accept(*(_to(torch, a, dev) for a in (p, q, d, u)))
    mxs.spec_kv_commit(t_len, n_emit, L)
    out = mxs.mxfp4_kv_dequant(t_nib, t_sc, t_len)
    torch.cuda.synchronize()

    # oracle chain
    lens = np.zeros(B, np.int32)
    oracle.kv_append(prompt, nib, sc, lens)
    lens = oracle.kv_commit(lens, lens0, L)
    oracle.kv_append(block, nib, sc, lens)
    _, n_ref, _, _ = oracle.spec_accept(p, q, d, u)
    lens = oracle.kv_commit(lens, n_ref, L)
    ref = oracle.kv_dequant(nib, sc, lens)

    assert np.array_equal(t_len.cpu().numpy(), lens)
    assert np.array_equal(out.cpu().numpy(), ref.astype(np.float32))
    assert np.all(lens == lens0 + n_ref) and n_ref.min() >= 1 and n_ref.max() <= T
