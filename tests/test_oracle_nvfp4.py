"""Pins of the NVFP4 oracle ("Module 11. Speculative Decoding and
Quantization", §12: E2M1 values in blocks of 16 sharing an E4M3 scale, one
FP32 scale per tensor, (16*4 + 8)/16 = 4.5 bits per value).

E4M3 is checked against an independent decoder (torch's float8_e4m3fn, a
library routine) and the format's closed-form landmarks; the dequantisation
and the GEMM against weights built here from the page's E2M1 magnitude table.
"""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _e2m1(code):
    return (-1.0 if code & 8 else 1.0) * E2M1[code & 7]


def test_e4m3_matches_an_independent_decoder():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_value(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and set(np.nonzero(nan)[0]) == {0x7F, 0xFF}
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_landmarks():
    assert oracle.e4m3_value(0x38) == 1.0          # exponent field = bias
    assert oracle.e4m3_value(0x7E) == 448.0        # largest finite
    assert oracle.e4m3_value(0x08) == 2.0 ** -6    # smallest normal
    assert oracle.e4m3_value(0x01) == 2.0 ** -9    # smallest subnormal
    assert oracle.e4m3_value(0x80) == 0.0 and oracle.e4m3_value(0xB8) == -1.0
    finite = {oracle.e4m3_value(c) for c in range(256) if c not in (0x7F, 0xFF)}
    assert len(finite) == 253                      # 254 finite codes, +0 and -0 equal


def test_bits_per_value_is_the_pages_figure():
    # [N, K/2] nibbles + [N, K/16] one-byte scales, per value
    N, K = 7, 4096
    bits = 8 * (N * K // 2 + N * K // 16) / (N * K)
    assert bits == (16 * 4 + 8) / 16 == 4.5


def _rand_nvfp4(N, K, seed):
    rng = np.random.default_rng(seed)
    nib = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    # finite positive and negative E4M3 scales, subnormals included
    sc = rng.integers(0, 0x7F, size=(N, K // 16)).astype(np.uint8)
    sc[rng.random(sc.shape) < 0.2] |= 0x80
    return nib, sc


def test_dequant_matches_table_construction():
    nib, sc = _rand_nvfp4(9, 64, 1)
    g = 0.37
    w = oracle.nvfp4_dequant(nib, sc, g)
    s = torch.from_numpy(sc).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for n in range(9):
        for k in range(64):
            code = (nib[n, k // 2] >> (4 * (k & 1))) & 15
            assert w[n, k] == _e2m1(code) * s[n, k // 16] * g


def test_gemm_matches_matmul_and_one_hot():
    nib, sc = _rand_nvfp4(33, 256, 2)
    x = workloads.bf16_normal(5, 256, seed=2)
    g = 2.0 ** -3 * 1.7
    y = oracle.nvfp4_gemm(x, nib, sc, g)
    xf = oracle.bf16_bits_to_f64(x)
    np.testing.assert_allclose(y, xf @ oracle.nvfp4_dequant(nib, sc, g).T, rtol=1e-12, atol=1e-12)
    # one-hot rows of X pick single weights
    eye = workloads.f32_to_bf16_bits(np.eye(256, dtype=np.float32)[[0, 17, 255]])
    y1 = oracle.nvfp4_gemm(eye, nib, sc, g)
    w = oracle.nvfp4_dequant(nib, sc, g)
    assert np.array_equal(y1, w[:, [0, 17, 255]].T)


def test_nan_scale_poisons_its_block_only():
    nib = np.full((2, 32), 0x22, np.uint8)  # code 2 = 1.0 everywhere
    sc = np.full((2, 4), 0x38, np.uint8)
    sc[1, 2] = 0x7F
    x = workloads.f32_to_bf16_bits(np.ones((1, 64), np.float32))
    y = oracle.nvfp4_gemm(x, nib, sc, 1.0)
    assert y[0, 0] == 64.0 and np.isnan(y[0, 1])
