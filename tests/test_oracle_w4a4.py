"""Pins for the oracle's W4A4 product, Y = dequant(pack(X)) . dequant(W)^T.

"Module 11. Speculative Decoding and Quantization", §12 names W4A4 (weights
and activations both 4-bit); the activation quantiser is the same block rule
as the weights' (§12-§13: one power-of-two scale per 32-element block, the
smallest one whose range holds the block maximum, nearest E2M1 value).  The
oracle composes ``pack`` (pinned in test_oracle_pack.py) with the plain
product (pinned in test_oracle_gemm.py); these tests pin the composition by
* hand-worked values of the rule: 5 rounds to 4 (tie, even fraction bit), 7
  in a block whose maximum is 7 takes scale 2 and rounds 3.5 to 4, i.e. 8;
* exactly representable activations, on which W4A4 equals the W4A16 product;
* sign symmetry and power-of-two scaling, which the rule keeps exactly;
* the error bound of the rule against the W4A16 product on random X;
* NaN rows (a non-finite activation) and NaN columns (a NaN weight scale).
"""
import json
import os

import numpy as np
import pytest

import oracle
import workloads

GOLD = os.path.join(os.path.dirname(__file__), "golden")
MAGS = [float(m) for m in json.load(open(os.path.join(GOLD, "e2m1_magnitudes.json")))["magnitudes"]]


def _bits(vals):
    return workloads.f32_to_bf16_bits(np.asarray(vals, dtype=np.float32))


def _ones_weights(N, K):
    # every weight 1.0: E2M1 code 2 in both nibbles, scale byte 127
    return np.full((N, K // 2), 0x22, dtype=np.uint8), np.full((N, K // 32), 127, dtype=np.uint8)


@pytest.mark.parametrize("v,want", [(5.0, 4.0), (-5.0, -4.0), (7.0, 8.0), (2.5, 2.0), (0.25, 0.25),
                                    (6.0, 6.0), (13.0, 12.0), (0.75, 0.75)])
def test_single_element_block_hand_worked(v, want):
    # one nonzero element per block: its block's scale is the smallest 2^e
    # with |v| <= 6 2^e; v 2^-e goes to the nearest E2M1 magnitude, ties to
    # the even fraction bit (5 -> 4, 3.5 -> 4, 2.5 -> 2; 13 takes scale 4: 3.25 -> 3)
    K = 64
    x = np.zeros((1, K), dtype=np.float32)
    x[0, 3] = v
    nib, sc = _ones_weights(2, K)
    y = oracle.gemm_w4a4(_bits(x), nib, sc)
    assert np.all(y == want)


def test_block_maximum_sets_the_scale_for_its_neighbours():
    # block max 12 -> scale 2: 12/2 = 6, 1/2 = 0.5, 0.6/2 = 0.3 -> 0.5, 0.2/2 -> 0
    K = 32
    x = np.zeros((1, K), dtype=np.float32)
    x[0, :4] = [12.0, 1.0, 0.6, 0.2]
    nib, sc = _ones_weights(1, K)
    assert oracle.gemm_w4a4(_bits(x), nib, sc)[0, 0] == 12.0 + 1.0 + 1.0 + 0.0


def test_representable_activations_equal_w4a16():
    rng = np.random.default_rng(11)
    M, N, K = 5, 7, 256
    grid = np.array(MAGS + [-m for m in MAGS])
    xv = grid[rng.integers(0, 16, size=(M, K))]
    e = rng.integers(-20, 21, size=(M, K // 32))
    xv = xv * np.repeat(2.0 ** e, 32, axis=1)
    xb = _bits(xv)
    assert np.all(oracle.bf16_bits_to_f64(xb) == xv)
    nib, sc = workloads.mxfp4_weights(N, K, 120, 134, seed=3, tensor_id=0)
    assert np.array_equal(oracle.gemm_w4a4(xb, nib, sc), oracle.gemm(xb, nib, sc))


def test_sign_symmetry_and_power_of_two_scaling():
    M, N, K = 4, 9, 320
    nib, sc = workloads.mxfp4_weights(N, K, 120, 134, seed=5, tensor_id=0)
    xb = workloads.bf16_normal(M, K, seed=5)
    y = oracle.gemm_w4a4(xb, nib, sc)
    xneg = xb ^ np.uint16(0x8000)
    assert np.array_equal(oracle.gemm_w4a4(xneg, nib, sc), -y)
    x = oracle.bf16_bits_to_f64(xb)
    for j in (-30, 7, 60):
        assert np.array_equal(oracle.gemm_w4a4(_bits(x * 2.0 ** j), nib, sc), y * 2.0 ** j)


def test_error_bound_against_w4a16():
    # |x - q(x)| <= 2^e per element (half the widest E2M1 gap, 4 -> 6, times
    # the block scale), so |Y_w4a4 - Y_w4a16| <= sum_k 2^e(k) |w[n, k]|; and
    # the rule is not the identity on N(0,1) data
    M, N, K = 6, 11, 512
    nib, sc = workloads.mxfp4_weights(N, K, 118, 132, seed=9, tensor_id=0)
    xb = workloads.bf16_normal(M, K, seed=9)
    x = oracle.bf16_bits_to_f64(xb)
    amax = np.abs(x.reshape(M, K // 32, 32)).max(axis=2)
    e = np.ceil(np.log2(amax / 6.0))
    step = np.repeat(2.0 ** e, 32, axis=1)
    w = oracle.dequant(nib, sc)
    bound = step @ np.abs(w).T
    d = np.abs(oracle.gemm_w4a4(xb, nib, sc) - oracle.gemm(xb, nib, sc))
    assert np.all(d <= bound)
    assert np.any(d > 0)


def test_nonfinite_activation_row_and_nan_scale_column():
    M, N, K = 4, 5, 96
    nib, sc = workloads.mxfp4_weights(N, K, 120, 134, seed=2, tensor_id=0)
    sc[3, 1] = 255
    xb = workloads.bf16_normal(M, K, seed=2)
    xb[1, 40] = 0x7F80  # +inf
    xb[2, 0] = 0x7FC0   # NaN
    y = oracle.gemm_w4a4(xb, nib, sc)
    assert np.all(np.isnan(y[1])) and np.all(np.isnan(y[2])) and np.all(np.isnan(y[:, 3]))
    good = np.ix_([0, 3], [0, 1, 2, 4])
    assert np.all(np.isfinite(y[good]))
    ref = oracle.gemm_w4a4(xb[[0, 3]], nib[[0, 1, 2, 4]], sc[[0, 1, 2, 4]])
    assert np.array_equal(y[good], ref)


def test_zero_and_subnormal_blocks():
    # an all-zero block contributes 0; a block of bf16 subnormals takes the
    # smallest scale 2^-127 and keeps values on its grid (0.5 2^-127 = 2^-128)
    K = 64
    x = np.zeros((2, K), dtype=np.float32)
    x[1, 32] = 2.0 ** -128
    x[1, 33] = 2.0 ** -127
    x[1, 34] = 3.0 * 2.0 ** -130  # 0.375 2^-127 -> 0.5 2^-127
    nib, sc = _ones_weights(1, K)
    y = oracle.gemm_w4a4(_bits(x), nib, sc)
    assert y[0, 0] == 0.0
    assert y[1, 0] == 2.0 ** -128 + 2.0 ** -127 + 2.0 ** -128
