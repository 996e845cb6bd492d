"""Pins of the MX-FP4 KV-cache oracle.

"Next-Gen Speculative Decoding and FP4 Quantization Shake Up LLM Inference
Economics" stores keys and values as MX-FP4 (its pipeline diagram's "KV Cache
Memory Pool (FP4)"; "Benchmarks and Real-World Impact", item 2: 62 % less KV
memory).  "Module 11. Speculative Decoding and Quantization" §4: after
acceptance the unaccepted suffix and its cache entries are discarded and
decoding continues from the corrected prefix.

Checked against rows built here from the page's E2M1 magnitude table (exact
round trips), brute-force placement and length arithmetic, and a worked
verification cycle.
"""
import numpy as np
import pytest

import oracle

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _grid_rows(shape, seed):
    """Rows whose every 32-block is exactly representable: E2M1 grid values
    times one power of two per block (and the block maximum 6 * 2^e, so the
    pack rule picks that e)."""
    rng = np.random.default_rng(seed)
    *lead, W = shape
    nb = W // 32
    mag = np.array(E2M1)[rng.integers(0, 8, size=(*lead, nb, 32))]
    mag[..., 0] = 6.0
    sign = np.where(rng.random((*lead, nb, 32)) < 0.5, -1.0, 1.0)
    e = rng.integers(-20, 20, size=(*lead, nb, 1))
    return (mag * sign * np.exp2(e)).reshape(shape).astype(np.float32)


def _cache(B, L, W, fill=0):
    return np.full((B, L, W // 2), fill, np.uint8), np.full((B, L, W // 32), fill, np.uint8)


def test_round_trip_at_the_committed_positions():
    B, T, L, W = 3, 5, 16, 256
    kv = _grid_rows((B, T, W), 1)
    nib, sc = _cache(B, L, W)
    lens = np.array([0, 7, 11], np.int32)
    assert oracle.kv_append(kv, nib, sc, lens) == 0
    out = oracle.kv_dequant(nib, sc, lens + T)
    for b in range(B):
        assert np.array_equal(out[b, lens[b]:lens[b] + T], kv[b].astype(np.float64))
        assert np.all(out[b, lens[b] + T:] == 0.0)


def test_only_the_block_positions_are_written():
    B, T, L, W = 4, 3, 10, 64
    rng = np.random.default_rng(2)
    kv = rng.standard_normal((B, T, W)).astype(np.float32)
    nib, sc = _cache(B, L, W, fill=0xAB)
    lens = rng.integers(0, L - T + 1, size=B).astype(np.int32)
    oracle.kv_append(kv, nib, sc, lens)
    pn, ps, _ = oracle.pack(kv.reshape(B * T, W))
    for b in range(B):
        for l in range(L):
            t = l - lens[b]
            if 0 <= t < T:
                assert np.array_equal(nib[b, l], pn[b * T + t]) and np.array_equal(sc[b, l], ps[b * T + t])
            else:
                assert np.all(nib[b, l] == 0xAB) and np.all(sc[b, l] == 0xAB)


def test_positions_past_the_cache_are_not_written():
    B, T, L, W = 3, 5, 8, 32
    kv = _grid_rows((B, T, W), 3)
    nib, sc = _cache(B, L, W, fill=0x11)
    lens = np.array([6, 8, 3], np.int32)  # 3 rows fit, none fit, all fit
    assert oracle.kv_append(kv, nib, sc, lens) == (T - 2) + T
    out = oracle.kv_dequant(nib, sc, np.full(B, L, np.int32))
    assert np.array_equal(out[0, 6:8], kv[0, :2].astype(np.float64))
    assert np.all(nib[1] == 0x11)
    assert np.array_equal(out[2, 3:8], kv[2].astype(np.float64))


def test_commit_brute_force():
    rng = np.random.default_rng(4)
    L = 50
    lens = rng.integers(0, L + 1, size=200).astype(np.int32)
    n = rng.integers(-2, 9, size=200).astype(np.int32)
    got = oracle.kv_commit(lens, n, L)
    for i in range(200):
        assert got[i] == min(int(lens[i]) + max(int(n[i]), 0), L)


def test_a_verification_cycle_discards_the_rejected_suffix():
    # 10 committed positions; the pass feeds the last committed token and 4
    # drafts (T = 5) into positions 10..14.  Drafts 1 and 2 are accepted, draft
    # 3 is rejected and replaced: 3 tokens emitted.  The entries of the last
    # committed token and the two accepted drafts (10, 11, 12) stay; those of
    # drafts 3 and 4 (13, 14) are the discarded suffix; the replacement token is
    # fed, and cached, by the next pass at position 13.
    L, W, T = 32, 64, 5
    nib, sc = _cache(1, L, W)
    prefix = _grid_rows((1, 10, W), 5)
    assert oracle.kv_append(prefix, nib, sc, np.array([0], np.int32)) == 0
    block = _grid_rows((1, T, W), 6)
    assert oracle.kv_append(block, nib, sc, np.array([10], np.int32)) == 0
    lens = oracle.kv_commit(np.array([10], np.int32), np.array([3], np.int32), L)
    assert lens[0] == 13
    out = oracle.kv_dequant(nib, sc, lens)
    assert np.array_equal(out[0, :10], prefix[0].astype(np.float64))
    assert np.array_equal(out[0, 10:13], block[0, :3].astype(np.float64))
    assert np.all(out[0, 13:] == 0.0)
    # the next pass overwrites the discarded entries from position 13 on
    nxt = _grid_rows((1, T, W), 7)
    oracle.kv_append(nxt, nib, sc, lens)
    out = oracle.kv_dequant(nib, sc, lens + T)
    assert np.array_equal(out[0, 13:18], nxt[0].astype(np.float64))
    # all drafts accepted plus the bonus token: the whole block stays
    assert oracle.kv_commit(np.array([10], np.int32), np.array([5], np.int32), L)[0] == 15
    # a refused row (0 tokens) commits nothing
    assert oracle.kv_commit(np.array([10], np.int32), np.array([0], np.int32), L)[0] == 10


def test_nonfinite_rows_follow_the_pack_rule():
    kv = np.ones((1, 2, 64), np.float32)
    kv[0, 1, 40] = np.nan
    nib, sc = _cache(1, 4, 64)
    oracle.kv_append(kv, nib, sc, np.array([1], np.int32))
    assert sc[0, 2, 1] == 255 and np.all(nib[0, 2, 16:32] == 0)
    out = oracle.kv_dequant(nib, sc, np.array([3], np.int32))
    assert np.all(np.isnan(out[0, 2, 32:])) and np.all(out[0, 2, :32] == 1.0)


def test_bf16_rows_convert_exactly():
    kv = _grid_rows((2, 3, 96), 8)
    bits = (kv.view(np.uint32) >> 16).astype(np.uint16)  # grid values are exact in bf16
    assert np.array_equal((bits.astype(np.uint32) << 16).view(np.float32), kv)
    n1, s1 = _cache(2, 6, 96)
    n2, s2 = _cache(2, 6, 96)
    lens = np.array([1, 3], np.int32)
    oracle.kv_append(kv, n1, s1, lens)
    oracle.kv_append(bits, n2, s2, lens, dtype="bf16")
    assert np.array_equal(n1, n2) and np.array_equal(s1, s2)


def test_footprint_is_below_the_pages_figure():
    # [W/2] nibble bytes + [W/32] scale bytes per position: 4.25 bits per value
    # against bf16's 16, a 73.4 % reduction; the page reports 62 % for its
    # whole KV memory (which also holds what this cache leaves out)
    W = 4096
    bits = 8 * (W // 2 + W // 32) / W
    assert bits == 4.25
    assert 1 - bits / 16 == pytest.approx(0.734375)
    assert 1 - bits / 16 >= 0.62
