"""Pins for the oracle's verification GEMM, Y = X . dequant(W)^T.

The method reaches exactly the plain definition (up to summation order), so
the oracle is that definition; it is pinned here by
* the hand-worked block example (tests/golden/dequant_hand_example.json);
* a closed form (constant code, constant scale, X = 1 -> Y = K * v * 2^(e-127));
* brute force: one-hot weights pick out single columns of X;
* a library special case: dense weights built by the test from the page's
  magnitude table, multiplied with numpy's float64 matmul.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import workloads

GOLD = os.path.join(os.path.dirname(__file__), "golden")
MAGS = json.load(open(os.path.join(GOLD, "e2m1_magnitudes.json")))["magnitudes"]
TABLE = np.array([float(m) for m in MAGS] + [-float(m) for m in MAGS], dtype=np.float64)  # code -> value


def _bf16_bits(vals):
    return workloads.f32_to_bf16_bits(np.asarray(vals, dtype=np.float32))


def _pack_codes(codes):
    """codes [N, K] (0..15) -> bytes [N, K/2], element 2i in the low nibble."""
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def test_hand_worked_block_dot():
    g = json.load(open(os.path.join(GOLD, "dequant_hand_example.json")))["block_dot"]
    nib = np.zeros((1, 16), dtype=np.uint8)
    nib[0, 0] = int(g["byte0"], 16)
    sc = np.array([[g["scale"]]], dtype=np.uint8)
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, :2] = g["x_prefix"]
    y = oracle.gemm(_bf16_bits(x), nib, sc)
    assert y[0, 0] == g["y"]


@pytest.mark.parametrize("code", range(16))
@pytest.mark.parametrize("e", [100, 127, 140])
def test_closed_form_constant_weights(code, e):
    K = 96
    nib = _pack_codes(np.full((3, K), code))
    sc = np.full((3, K // 32), e, dtype=np.uint8)
    x = _bf16_bits(np.ones((2, K)))
    y = oracle.gemm(x, nib, sc)
    assert np.all(y == K * TABLE[code] * 2.0 ** (e - 127))


def test_one_hot_weights_select_columns():
    rng = np.random.default_rng(7)
    M, K = 3, 64
    xf = rng.standard_normal((M, K)).astype(np.float32)
    xb = _bf16_bits(xf)
    xv = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for k in (0, 1, 31, 32, 63):
        for code in (1, 7, 9, 15):
            codes = np.zeros((1, K), dtype=np.uint8)
            codes[0, k] = code
            sc = np.array([[127, 129]], dtype=np.uint8)
            y = oracle.gemm(xb, _pack_codes(codes), sc)
            expect = xv[:, k] * TABLE[code] * 2.0 ** (sc[0, k // 32] - 127)
            assert np.array_equal(y[:, 0], expect)


def test_matches_library_matmul_on_test_built_weights():
    rng = np.random.default_rng(11)
    M, N, K = 5, 37, 256
    codes = rng.integers(0, 16, size=(N, K))
    exps = rng.integers(110, 140, size=(N, K // 32)).astype(np.uint8)
    wd = TABLE[codes] * np.repeat(2.0 ** (exps.astype(np.float64) - 127), 32, axis=1)
    xb = _bf16_bits(rng.standard_normal((M, K)))
    xv = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    y = oracle.gemm(xb, _pack_codes(codes), exps, nthreads=3)
    ref = xv @ wd.T
    assert np.max(np.abs(y - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_nan_scale_poisons_only_its_rows():
    nib = _pack_codes(np.full((2, 32), 2))
    sc = np.array([[255], [127]], dtype=np.uint8)
    y = oracle.gemm(_bf16_bits(np.ones((1, 32))), nib, sc)
    assert math.isnan(y[0, 0]) and y[0, 1] == 32.0


def test_thread_count_does_not_change_result():
    x, nib, sc = workloads.tiny_gemm_inputs(0)
    y1 = oracle.gemm(x, nib, sc, nthreads=1)
    y7 = oracle.gemm(x, nib, sc, nthreads=7)
    assert np.array_equal(y1, y7)
