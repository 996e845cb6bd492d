"""Pins for the oracle's element decode (E2M1, E8M0) and dequantisation.

Pinned against the pages, not against the oracle itself:
* the E2M1 magnitude set and the 16-encodings / 15-values count printed in
  "Module 11. Speculative Decoding and Quantization", §12;
* a hand-worked decode example (tests/golden/dequant_hand_example.json);
* IEEE-style monotone encoding: the 8 non-negative codes, read as integers,
  list the magnitudes in ascending order.
"""
import json
import math
import os

import numpy as np

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def test_e2m1_magnitude_set_and_count():
    g = _gold("e2m1_magnitudes.json")
    vals = [oracle.e2m1_value(c) for c in range(16)]
    assert sorted({abs(v) for v in vals}) == g["magnitudes"]
    # 16 encodings, 15 distinct values: +0 and -0 coincide
    assert len(vals) == g["encodings"]
    assert len(set(vals)) == g["distinct_values"]
    assert math.copysign(1.0, vals[8]) == -1.0 and vals[8] == 0.0


def test_e2m1_monotone_encoding_and_sign_bit():
    mags = _gold("e2m1_magnitudes.json")["magnitudes"]
    for c in range(8):
        assert oracle.e2m1_value(c) == mags[c]
        assert oracle.e2m1_value(c | 8) == -mags[c]


def test_e8m0_power_of_two():
    assert oracle.e8m0_value(127) == 1.0
    assert oracle.e8m0_value(126) == 0.5
    assert oracle.e8m0_value(133) == 64.0
    assert oracle.e8m0_value(0) == 2.0 ** -127
    assert oracle.e8m0_value(254) == 2.0 ** 127
    assert math.isnan(oracle.e8m0_value(255))
    # no fraction field: every value is an exact power of two
    for e in range(255):
        m, _ = math.frexp(oracle.e8m0_value(e))
        assert m == 0.5


def test_bits_per_value_accounting():
    g = _gold("e2m1_magnitudes.json")
    blk = g["mx_block"]
    assert (blk * 4 + 8) / blk == g["mxfp4_bits_per_value"]
    assert (16 * 4 + 8) / 16 == g["nvfp4_bits_per_value"]
    # the packed buffers hold exactly N*K/2 + N*K/32 bytes = 4.25 bits/value
    N, K = 256, 512
    assert (N * K // 2 + N * K // 32) * 8 / (N * K) == g["mxfp4_bits_per_value"]


def test_hand_worked_dequant_pairs():
    g = _gold("dequant_hand_example.json")
    for case in g["cases"]:
        nib = np.zeros((1, 16), dtype=np.uint8)
        nib[0, 0] = int(case["byte"], 16)
        sc = np.array([[case["scale"]]], dtype=np.uint8)
        w = oracle.dequant(nib, sc)
        assert w[0, 0] == case["pair"][0]
        assert w[0, 1] == case["pair"][1]
        assert math.copysign(1.0, w[0, 1]) == math.copysign(1.0, case["pair"][1])
        assert np.all(w[0, 2:] == 0.0)


def test_dequant_block_scale_applies_per_32():
    # two blocks with different scales: each scale covers exactly 32 elements
    nib = np.full((1, 32), 0x22, dtype=np.uint8)  # every element code 2 -> 1.0
    sc = np.array([[127, 130]], dtype=np.uint8)
    w = oracle.dequant(nib, sc)
    assert np.all(w[0, :32] == 1.0) and np.all(w[0, 32:] == 8.0)
