"""Pins for the oracle's MXFP4 pack (real weights -> nibbles + E8M0 scales).

The pages fix the grid and the block structure ("Module 11 ...", §12) and show
a teaching quantizer that uses one scale per group and scale 1 for an
all-zero group (§13).  The power-of-two scale choice (smallest e with
amax <= 6 * 2^e) and ties-to-even are this build's stated readings; they are
pinned by brute force over every code and scale, by the round-trip bound, and
by explicit tie cases.
"""
import json
import os

import numpy as np

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")
MAGS = json.load(open(os.path.join(GOLD, "e2m1_magnitudes.json")))["magnitudes"]
TABLE = np.array([float(m) for m in MAGS] + [-float(m) for m in MAGS], dtype=np.float64)


def _unpack(nib):
    out = np.empty((nib.shape[0], nib.shape[1] * 2), dtype=np.int64)
    out[:, 0::2] = nib & 15
    out[:, 1::2] = nib >> 4
    return out


def _values(nib, sc):
    return TABLE[_unpack(nib)] * np.repeat(2.0 ** (sc.astype(np.float64) - 127), 32, axis=1)


def test_zero_block_gets_scale_one_and_zero_codes():
    nib, sc, ok = oracle.pack(np.zeros((2, 64), dtype=np.float32))
    assert ok and np.all(sc == 127) and np.all(nib == 0)


def test_negative_zero_keeps_sign_bit():
    w = np.zeros((1, 32), dtype=np.float32)
    w[0, 3] = -0.0
    w[0, 5] = 6.0
    w[0, 6] = -1e-6  # rounds to zero, sign kept
    nib, sc, ok = oracle.pack(w)
    codes = _unpack(nib)[0]
    assert codes[3] == 8 and codes[6] == 8 and codes[5] == 7 and sc[0, 0] == 127


def test_brute_force_every_code_and_scale_roundtrips():
    # a block holding the full-magnitude code 7 (value 6) fixes the scale, so
    # every other code in the block must come back unchanged
    for e in (1, 60, 120, 127, 133, 200, 252):  # 6 * 2^(e-127) must be a finite fp32
        codes = np.tile(np.arange(16), 2)[None, :].copy()
        codes[0, 0] = 7
        vals = TABLE[codes] * 2.0 ** (e - 127)
        nib, sc, ok = oracle.pack(vals.astype(np.float32))
        assert ok
        assert sc[0, 0] == e
        assert np.array_equal(_unpack(nib), codes)


def test_value_roundtrip_on_representable_blocks():
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 16, size=(64, 128))
    exps = rng.integers(100, 150, size=(64, 4))
    vals = TABLE[codes] * np.repeat(2.0 ** (exps - 127.0), 32, axis=1)
    nib, sc, ok = oracle.pack(vals.astype(np.float32))
    assert ok
    assert np.array_equal(_values(nib, sc), vals)


def test_smallest_scale_covers_block_max():
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((32, 256)) * 10.0 ** rng.uniform(-6, 6, size=(32, 1))).astype(np.float32)
    nib, sc, ok = oracle.pack(w)
    blocks = np.abs(w.astype(np.float64)).reshape(32, 8, 32).max(axis=2)
    s = 2.0 ** (sc.astype(np.float64) - 127)
    assert np.all(blocks <= 6 * s)
    assert np.all(blocks > 3 * s)  # one exponent lower would not cover amax


def test_roundtrip_error_within_half_grid_step():
    rng = np.random.default_rng(9)
    w = rng.standard_normal((16, 512)).astype(np.float32)
    nib, sc, ok = oracle.pack(w)
    back = _values(nib, sc)
    s = np.repeat(2.0 ** (sc.astype(np.float64) - 127), 32, axis=1)
    a = np.abs(w.astype(np.float64)) / s
    half_step = np.where(a <= 2, 0.25, np.where(a <= 4, 0.5, 1.0))
    assert np.all(np.abs(back - w) <= half_step * s)


def test_ties_go_to_even_fraction_bit():
    # midpoints between neighbouring grid values, block scale fixed at 1 by a 6
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    expect = [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]
    w = np.zeros((1, 32), dtype=np.float32)
    w[0, 0] = 6.0
    w[0, 1:8] = mids
    w[0, 8:15] = [-m for m in mids]
    nib, sc, ok = oracle.pack(w)
    vals = _values(nib, sc)[0]
    assert sc[0, 0] == 127
    assert list(vals[1:8]) == expect
    assert list(vals[8:15]) == [-v for v in expect]


def test_nonfinite_block_is_flagged():
    w = np.ones((1, 64), dtype=np.float32)
    w[0, 40] = np.inf
    nib, sc, ok = oracle.pack(w)
    assert not ok and sc[0, 1] == 255 and np.all(nib[0, 16:] == 0) and sc[0, 0] == 125


def test_bf16_input_matches_fp32_of_same_values():
    rng = np.random.default_rng(2)
    w = rng.standard_normal((4, 64)).astype(np.float32)
    bits = (w.view(np.uint32) >> 16).astype(np.uint16)  # truncation: exact bf16 values
    wf = (bits.astype(np.uint32) << 16).view(np.float32)
    a = oracle.pack(bits, dtype="bf16")
    b = oracle.pack(wf)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
