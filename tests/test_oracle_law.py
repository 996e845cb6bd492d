"""Pins of the sampling-law oracle ("Module 11. Speculative Decoding and
Quantization", §4: acceptance uses the laws tokens are actually sampled from,
after temperature, top-k and top-p).

Each check is independent of the oracle's own steps: brute force over every
subset of a tiny vocabulary for "the smallest set of the most probable tokens
reaching mass p", counting for top-k, closed forms for two tokens, and
invariants (scaling by the temperature, normalisation, masked tokens).
"""
import itertools
import math

import numpy as np
import pytest

import oracle


def _softmax(z):
    z = np.asarray(z, dtype=np.float64)
    e = np.exp(z - z.max())
    return e / e.sum()


def _brute_law(l, T, k, p):
    """Transformed law by enumeration: top-k by counting larger logits, then
    the smallest subset (over all subsets) of the top-k law with mass >= p."""
    V = len(l)
    l64 = np.asarray(l, dtype=np.float64)
    keep = [t for t in range(V) if k <= 0 or k >= V or sum(l64[u] > l64[t] for u in range(V)) < k]
    base = np.zeros(V)
    base[keep] = _softmax(l64[keep] / T)
    if p < 1.0:
        best = None
        for size in range(1, len(keep) + 1):
            for sub in itertools.combinations(keep, size):
                m = base[list(sub)].sum()
                if m >= p and (best is None or m > best[0]):
                    best = (m, sub)
            if best is not None:
                break
        keep = list(best[1])
    out = np.zeros(V)
    out[keep] = base[keep] / base[keep].sum()
    return out


@pytest.mark.parametrize("seed", range(40))
def test_law_matches_brute_force_on_tiny_vocabularies(seed):
    rng = np.random.default_rng(seed)
    V = int(rng.integers(2, 8))
    l = (rng.standard_normal(V) * 2.0).astype(np.float32)
    T = float(rng.choice([0.3, 0.7, 1.0, 1.8]))
    k = int(rng.integers(0, V + 1))
    p = float(rng.choice([0.2, 0.5, 0.8, 0.95, 1.0]))
    got, margin, kept = oracle.sampling_law(l[None], T, k, p)
    ref = _brute_law(l, T, k, p)
    # the brute force picks the same set unless the cut sits on the boundary
    if margin[0] > 1e-12:
        np.testing.assert_allclose(got[0], ref, rtol=1e-12, atol=1e-15)
        assert kept[0] == np.count_nonzero(ref)


def test_two_tokens_closed_form():
    # no filters: p(first) = 1 / (1 + exp(-(l1 - l2) / T))
    for l1, l2, T in [(1.0, 0.0, 1.0), (3.5, -2.0, 0.5), (-1.25, 4.0, 2.0)]:
        got, _, _ = oracle.sampling_law(np.array([[l1, l2]], np.float32), T)
        assert got[0, 0] == pytest.approx(1.0 / (1.0 + math.exp(-(l1 - l2) / T)), rel=1e-14)


def test_temperature_scales_the_logits():
    rng = np.random.default_rng(1)
    l = rng.standard_normal((3, 50)).astype(np.float32)
    a, _, _ = oracle.sampling_law(l, 2.0)
    b, _, _ = oracle.sampling_law((l.astype(np.float64) / 2.0).astype(np.float32), 1.0)
    # l / 2 is exact in fp32 (a power of two)
    np.testing.assert_allclose(a, b, rtol=1e-14)


def test_top_k_one_and_tiny_top_p_give_the_argmax():
    rng = np.random.default_rng(2)
    l = rng.standard_normal((5, 200)).astype(np.float32)
    for kw in ({"top_k": 1}, {"top_p": 1e-9}):
        got, _, kept = oracle.sampling_law(l, 0.8, **kw)
        assert np.all(kept == 1)
        assert np.array_equal(np.argmax(got, axis=1), np.argmax(l, axis=1))
        assert np.all(got.max(axis=1) == 1.0)


def test_ties_at_the_top_k_boundary_are_kept():
    l = np.array([[3.0, 1.0, 2.0, 2.0, 0.0]], np.float32)
    got, _, kept = oracle.sampling_law(l, 1.0, top_k=2)
    assert kept[0] == 3 and got[0, 1] == 0.0 and got[0, 4] == 0.0
    assert got[0, 2] == got[0, 3]


def test_normalised_monotone_and_masked():
    rng = np.random.default_rng(3)
    l = rng.standard_normal((4, 300)).astype(np.float32)
    l[:, ::7] = -np.inf
    got, _, kept = oracle.sampling_law(l, 0.9, top_k=100, top_p=0.9)
    assert np.allclose(got.sum(axis=1), 1.0, rtol=0, atol=1e-13)
    assert np.all(got[:, ::7] == 0.0)
    for r in range(4):
        kept_idx = np.nonzero(got[r])[0]
        dropped = np.setdiff1d(np.arange(300), kept_idx)
        # what is kept is a top set: every kept logit beats every dropped one
        assert l[r, kept_idx].min() > l[r, dropped].max()
        # the top-p set is the smallest that reaches p under the top-k law
        base, _, _ = oracle.sampling_law(l[r:r + 1], 0.9, top_k=100)
        mass = np.sort(base[0])[::-1].cumsum()
        assert kept[r] == np.searchsorted(mass, 0.9) + 1


def test_rows_without_a_law():
    l = np.array([[np.nan, 0.0], [np.inf, 0.0], [-np.inf, -np.inf]], np.float32)
    got, _, kept = oracle.sampling_law(l)
    assert np.all(got == 0.0) and np.all(kept == 0)


def _chi2(counts, probs):
    m = probs > 0
    e = counts.sum() * probs[m]
    return float(((counts[m] - e) ** 2 / e).sum()) + (1e9 if counts[~m].sum() else 0.0)


def test_acceptance_on_transformed_laws_preserves_the_transformed_target():
    """§4: with the target and the draft both filtered the same way, the first
    emitted token follows the filtered target law; acceptance on the raw
    target law while drafts come from the filtered draft law does not."""
    rng = np.random.default_rng(11)
    V, B = 8, 1_000_000
    tl = (rng.standard_normal((2, V)) * 1.5).astype(np.float32)
    dl = (tl[:1] + rng.standard_normal((1, V)) * 0.8).astype(np.float32)
    T, k, p = 0.8, 6, 0.9
    pt, _, _ = oracle.sampling_law(tl, T, k, p)
    qt, _, _ = oracle.sampling_law(dl, T, k, p)
    assert np.count_nonzero(pt[0]) < V  # the filters do remove tokens
    c = np.cumsum(qt[0])
    draft = np.minimum(np.searchsorted(c, rng.random(B) * c[-1], side="right"), V - 1).astype(np.int32)[:, None]
    u = rng.random((B, 2))
    pb = np.broadcast_to(pt[None], (B, 2, V))
    qb = np.broadcast_to(qt[None], (B, 1, V))
    tok, _, _, _ = oracle.spec_accept(pb, qb, draft, u, f64=True)
    crit = 24.322  # chi-square critical value at p = 1e-3 for 7 degrees of freedom (at most 7 here)
    assert _chi2(np.bincount(tok[:, 0], minlength=V), pt[0]) < crit
    # planted mistake: the raw (unfiltered) target law in the test
    raw, _, _ = oracle.sampling_law(tl, 1.0)
    tok2, _, _, _ = oracle.spec_accept(np.broadcast_to(raw[None], (B, 2, V)), qb, draft, u, f64=True)
    assert _chi2(np.bincount(tok2[:, 0], minlength=V), pt[0]) > 100 * crit
