"""Pins for the oracle's acceptance / residual / bonus sampling.

Everything here is fixed by "Module 11. Speculative Decoding and
Quantization":
* §5 worked example A (alpha = 0.85 = 1 - TV, r = (1,0,0,0,0), balance = p);
* §5 block B18: Monte Carlo (12000 draws, max |freq - p| < 0.02), the tiny
  residual case, the zero-draw case, strict "<";
* §4 mass balance: accept/correct reproduces the target law -- checked by
  chi-square over 10^6 seeded trials at vocab 8 (first token, and the joint of
  the first two tokens with a continuation cycle), and by deterministic
  quadrature over the uniform on V = 2..4 (brute force);
* §4 boundaries: p = q never rejects; q(x) = 0 is a rejection;
* §6-§7 expected emitted tokens (closed form and the two-rate tail sum).
A planted mistake (emitting the draft law q instead of the corrected law) is
shown to fail the chi-square, so the statistic has power.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _sample(rng, law, size):
    """Inverse-CDF draws from a 1-D law (test-side input generation)."""
    c = np.cumsum(np.asarray(law, dtype=np.float64))
    return np.minimum(np.searchsorted(c, rng.random(size) * c[-1], side="right"),
                      len(law) - 1).astype(np.int32)


def _batch(p_laws, q_laws, B, rng, dtype=np.float32):
    """B rows sharing the same per-position laws; drafts x_i ~ q_i."""
    p_laws = np.asarray(p_laws, dtype=np.float64)
    q_laws = np.asarray(q_laws, dtype=np.float64).reshape(-1, p_laws.shape[1])
    K = q_laws.shape[0]
    p = np.broadcast_to(p_laws.astype(dtype), (B,) + p_laws.shape)
    q = np.broadcast_to(q_laws.astype(dtype), (B,) + q_laws.shape)
    draft = np.stack([_sample(rng, q_laws[i], B) for i in range(K)], axis=1) if K else np.zeros((B, 0), np.int32)
    u = rng.random((B, K + 1)).astype(dtype)
    return p, q, draft, u


def _chi2(counts, probs):
    n = counts.sum()
    e = n * np.asarray(probs, dtype=np.float64)
    return float(((counts - e) ** 2 / e).sum())


# chi-square critical values at p = 1e-3 (7 and 63 degrees of freedom)
CHI2_7 = 24.322
CHI2_63 = 103.442


def test_closed_form_expected_tokens_matches_printed_values():
    g = _gold("expected_tokens.json")
    for c in g["closed_form"]:
        a, gam = c["alpha"], c["gamma"]
        assert round((1 - a ** (gam + 1)) / (1 - a), 2) == c["E"]
        assert round(sum(a ** k for k in range(gam + 1)), 2) == c["E"]
    r = g["tail_sum"]["rates"]
    assert round(1 + r[0] + r[0] * r[1], 2) == g["tail_sum"]["E"]
    m = sum(r) / 2
    assert round(1 + m + m * m, 2) == g["tail_sum"]["E_at_mean_rate"]


def test_worked_example_a_by_quadrature():
    """Exact enumeration over x ~ q and a midpoint grid over u."""
    g = _gold("worked_example_a.json")
    pA, qA = np.array(g["p"]), np.array(g["q"])
    V, G = 5, 20000
    xs = np.repeat(np.arange(V, dtype=np.int32), G)
    u0 = np.tile((np.arange(G) + 0.5) / G, V)
    B = V * G
    p = np.broadcast_to(np.stack([pA, pA]), (B, 2, V))
    q = np.broadcast_to(qA[None, :], (B, 1, V))
    u = np.stack([u0, np.full(B, 0.37)], axis=1)
    tok, n, flags, _ = oracle.spec_accept(p, q, xs[:, None], u, f64=True)
    w = np.repeat(qA, G) / G  # weight of each (x, u) cell
    alpha = float((w * (n == 2)).sum())
    assert abs(alpha - g["alpha"]) <= 2.0 / G
    assert abs(alpha - (1 - 0.5 * np.abs(pA - qA).sum())) <= 2.0 / G  # alpha = 1 - TV
    # every rejection samples the residual r = (1,0,0,0,0)
    assert np.all(tok[n == 1, 0] == int(np.argmax(g["r"])))
    # balance: the law of the emitted token is p
    law = np.array([(w * (tok[:, 0] == t)).sum() for t in range(V)])
    assert np.max(np.abs(law - pA)) <= 2.0 / G


def test_b18_monte_carlo():
    g = _gold("b18_checks.json")["monte_carlo"]
    wa = _gold("worked_example_a.json")
    pA, qA = np.array(wa["p"]), np.array(wa["q"])
    rng = np.random.default_rng(18)
    p, q, d, u = _batch([pA, pA], [qA], g["draws"], rng, dtype=np.float64)
    tok, n, _, _ = oracle.spec_accept(p, q, d, u, f64=True)
    freq = np.bincount(tok[:, 0], minlength=5) / g["draws"]
    assert np.max(np.abs(freq - pA)) < g["max_abs_freq_err"]


def test_b18_tiny_residual_stays_a_distribution():
    g = _gold("b18_checks.json")["tiny_residual"]
    p0 = np.array([1.0 - 1e-14, 1e-14])
    q0 = np.array(g["q"])
    # reject the proposal 0 (u * 1 >= 1 - 1e-14), then sample the residual
    for u1 in (0.0, 0.5, 0.999999):
        p = np.stack([p0, p0])[None]
        q = q0[None, None, :]
        u = np.array([[1.0 - 1e-15, u1]])
        tok, n, flags, _ = oracle.spec_accept(p, q, np.array([[0]], np.int32), u, f64=True)
        assert n[0] == 1 and tok[0, 0] == int(np.argmax(g["r"])) and flags[0] == 0


def test_b18_zero_draw_rejects_zero_acceptance():
    g = _gold("b18_checks.json")["zero_draw"]
    p0, q0 = np.array(g["p"]), np.array(g["q"])
    for dt in (True, False):
        p = np.stack([p0, p0])[None]
        q = q0[None, None, :]
        u = np.array([[g["draw"], 0.5]])
        tok, n, flags, _ = oracle.spec_accept(p, q, np.array([[g["proposal"]]], np.int32), u, f64=dt)
        assert tok[0, 0] == g["token"] and n[0] == 1  # rejected, residual token


def test_strict_less_than_at_equality():
    # u * q(x) == p(x) exactly must reject (draw < acceptance is strict)
    p = np.array([[[0.25, 0.75], [0.5, 0.5]]], np.float32)
    q = np.array([[[0.5, 0.5]]], np.float32)
    u = np.array([[0.5, 0.0]], np.float32)  # 0.5 * 0.5 == 0.25
    tok, n, _, _ = oracle.spec_accept(p, q, np.array([[0]], np.int32), u)
    assert n[0] == 1 and tok[0, 0] == 1
    u = np.array([[np.nextafter(np.float32(0.5), np.float32(0)), 0.0]], np.float32)
    tok, n, _, _ = oracle.spec_accept(p, q, np.array([[0]], np.int32), u)
    assert n[0] == 2 and tok[0, 0] == 0


def test_p_equals_q_never_rejects_and_bonus_comes_from_p():
    rng = np.random.default_rng(4)
    V, K, B = 8, 5, 40000
    law = rng.dirichlet(np.ones(V))
    bonus = rng.dirichlet(np.ones(V))
    p, q, d, u = _batch(np.vstack([np.tile(law, (K, 1)), bonus]), np.tile(law, (K, 1)), B, rng)
    tok, n, flags, _ = oracle.spec_accept(p, q, d, u)
    assert np.all(n == K + 1) and np.all(flags == 0)
    assert np.array_equal(tok[:, :K], d)
    counts = np.bincount(tok[:, K], minlength=V)
    assert _chi2(counts, bonus.astype(np.float32).astype(np.float64) / bonus.astype(np.float32).sum()) < CHI2_7


def test_zero_q_proposal_is_rejected_and_flagged():
    p = np.array([[[0.5, 0.5], [0.5, 0.5]]], np.float32)
    q = np.array([[[0.0, 1.0]]], np.float32)
    u = np.array([[0.0, 0.1]], np.float32)
    tok, n, flags, _ = oracle.spec_accept(p, q, np.array([[0]], np.int32), u)
    assert n[0] == 1 and flags[0] & oracle.ROW_ZERO_Q and tok[0, 0] == 0


def test_bad_draft_id_marks_row():
    p = np.full((2, 3, 4), 0.25, np.float32)
    q = np.full((2, 2, 4), 0.25, np.float32)
    d = np.array([[0, 4], [1, 2]], np.int32)
    u = np.zeros((2, 3), np.float32)
    tok, n, flags, _ = oracle.spec_accept(p, q, d, u)
    assert n[0] == 0 and flags[0] & oracle.ROW_BAD_DRAFT and np.all(tok[0] == -1)
    assert n[1] == 3 and flags[1] == 0


def test_zero_residual_falls_back_to_p():
    # unnormalised inputs: p(x) < q(x) everywhere, so (p - q)+ = 0
    p = np.array([[[0.2, 0.3], [0.9, 0.1]]], np.float32)
    q = np.array([[[0.5, 0.5]]], np.float32)
    for u1, expect in ((0.1, 0), (0.7, 1)):
        u = np.array([[0.9, u1]], np.float32)
        tok, n, flags, _ = oracle.spec_accept(p, q, np.array([[0]], np.int32), u)
        assert n[0] == 1 and flags[0] & oracle.ROW_ZERO_RESIDUAL and tok[0, 0] == expect


def test_all_zero_law_is_an_error_row():
    p = np.zeros((1, 1, 4), np.float32)
    q = np.zeros((1, 0, 4), np.float32)
    tok, n, flags, _ = oracle.spec_accept(p, q, np.zeros((1, 0), np.int32), np.zeros((1, 1), np.float32))
    assert n[0] == 0 and flags[0] & oracle.ROW_NONFINITE


def test_no_drafts_samples_bonus_only():
    rng = np.random.default_rng(8)
    V, B = 8, 200000
    law = rng.dirichlet(np.ones(V))
    p, q, d, u = _batch(law[None], np.zeros((0, V)), B, rng)
    tok, n, _, _ = oracle.spec_accept(p, q, d, u)
    assert np.all(n == 1)
    lf = law.astype(np.float32).astype(np.float64)
    assert _chi2(np.bincount(tok[:, 0], minlength=V), lf / lf.sum()) < CHI2_7


def _vocab8_laws(seed):
    rng = np.random.default_rng(seed)
    p = rng.dirichlet(np.ones(8) * 0.7, size=4)
    q = rng.dirichlet(np.ones(8) * 0.7, size=4)
    return p, q


def test_chi_square_first_token_is_target_law():
    p_laws, q_laws = _vocab8_laws(100)
    rng = np.random.default_rng(101)
    B = 1_000_000
    p, q, d, u = _batch(p_laws[:2], q_laws[:1], B, rng, dtype=np.float64)
    tok, n, _, _ = oracle.spec_accept(p, q, d, u, f64=True)
    counts = np.bincount(tok[:, 0], minlength=8)
    assert _chi2(counts, p_laws[0]) < CHI2_7
    # planted mistake: emitting the draft token unconditionally gives law q
    wrong = np.bincount(d[:, 0], minlength=8)
    assert _chi2(wrong, p_laws[0]) > 100 * CHI2_7


def test_chi_square_joint_of_two_tokens_with_continuation():
    """Two emitted tokens of history-independent laws p_1, p_2 must be
    distributed as p_1 x p_2; a cycle that emits one token is continued by a
    second cycle that starts at position 2."""
    p_laws, q_laws = _vocab8_laws(200)
    rng = np.random.default_rng(201)
    B = 1_000_000
    p, q, d, u = _batch(p_laws[:3], q_laws[:2], B, rng, dtype=np.float64)
    tok, n, _, _ = oracle.spec_accept(p, q, d, u, f64=True)
    first = tok[:, 0].copy()
    second = tok[:, 1].copy()
    short = np.nonzero(n == 1)[0]
    p2, q2, d2, u2 = _batch(p_laws[1:4], q_laws[1:3], len(short), rng, dtype=np.float64)
    tok2, _, _, _ = oracle.spec_accept(p2, q2, d2, u2, f64=True)
    second[short] = tok2[:, 0]
    counts = np.bincount(first * 8 + second, minlength=64)
    assert _chi2(counts, np.outer(p_laws[0], p_laws[1]).ravel()) < CHI2_63


@pytest.mark.parametrize("V", [2, 3, 4])
@pytest.mark.parametrize("K", [1, 2])
def test_brute_force_law_by_quadrature(V, K):
    """Exact enumeration of every draft sequence x (weight prod q_i(x_i)) and a
    midpoint grid over each uniform; the emitted first token must follow p_1
    to quadrature accuracy."""
    rng = np.random.default_rng(300 + 10 * V + K)
    p_laws = rng.dirichlet(np.ones(V), size=K + 1)
    q_laws = rng.dirichlet(np.ones(V), size=K)
    q_laws[0, 0] = 0.0  # include a zero-mass proposal token
    q_laws[0] /= q_laws[0].sum()
    G = 64
    grid = (np.arange(G) + 0.5) / G
    seqs = np.array(np.meshgrid(*[np.arange(V)] * K, indexing="ij")).reshape(K, -1).T
    ugrid = np.array(np.meshgrid(*[grid] * (K + 1), indexing="ij")).reshape(K + 1, -1).T
    rows_x = np.repeat(seqs, len(ugrid), axis=0).astype(np.int32)
    rows_u = np.tile(ugrid, (len(seqs), 1))
    wx = np.prod([q_laws[i][seqs[:, i]] for i in range(K)], axis=0)
    w = np.repeat(wx, len(ugrid)) / len(ugrid)
    B = len(rows_x)
    p = np.broadcast_to(p_laws, (B,) + p_laws.shape)
    q = np.broadcast_to(q_laws, (B,) + q_laws.shape)
    tok, n, _, _ = oracle.spec_accept(p, q, rows_x, rows_u, f64=True)
    law = np.array([(w * (tok[:, 0] == t)).sum() for t in range(V)])
    assert abs(law.sum() - 1.0) < 1e-12
    assert np.max(np.abs(law - p_laws[0])) <= 2.0 / G


def _constant_overlap_laws(alpha, V, rng):
    """q with q(t0) = 0 and p = alpha * q + (1 - alpha) * e_t0, so that
    sum_t min(p_t, q_t) = alpha exactly."""
    q = rng.dirichlet(np.ones(V))
    q[0] = 0.0
    q /= q.sum()
    p = alpha * q
    p[0] += 1.0 - alpha
    return p, q


@pytest.mark.parametrize("alpha,gamma,printed", [(0.7, 5, 2.94), (0.9, 7, 5.70), (0.85, 4, 3.71)])
def test_mean_emitted_matches_closed_form(alpha, gamma, printed):
    rng = np.random.default_rng(int(alpha * 100) + gamma)
    p1, q1 = _constant_overlap_laws(alpha, 8, rng)
    assert abs(np.minimum(p1, q1).sum() - alpha) < 1e-12
    B = 200_000
    p, q, d, u = _batch(np.tile(p1, (gamma + 1, 1)), np.tile(q1, (gamma, 1)), B, rng, dtype=np.float64)
    _, n, _, _ = oracle.spec_accept(p, q, d, u, f64=True)
    E = (1 - alpha ** (gamma + 1)) / (1 - alpha)
    se = n.std() / np.sqrt(B)
    assert abs(n.mean() - E) < 5 * se
    assert round(E, 2) == printed


def test_two_rate_tail_sum():
    rng = np.random.default_rng(77)
    pa, qa = _constant_overlap_laws(0.9, 8, rng)
    pb, qb = _constant_overlap_laws(0.5, 8, rng)
    B = 400_000
    p, q, d, u = _batch(np.vstack([pa, pb, pb]), np.vstack([qa, qb]), B, rng, dtype=np.float64)
    _, n, _, _ = oracle.spec_accept(p, q, d, u, f64=True)
    se = n.std() / np.sqrt(B)
    assert abs(n.mean() - 2.35) < 5 * se
    assert abs(n.mean() - 2.19) > 20 * se  # the mean rate alone is not enough


def test_edge_distance_reported():
    p = np.array([[[0.5, 0.5]]], np.float64)
    q = np.zeros((1, 0, 2))
    tok, n, _, edge = oracle.spec_accept(p, q, np.zeros((1, 0), np.int32), np.array([[0.5 + 1e-7]]), f64=True)
    assert tok[0, 0] == 1 and abs(edge[0] - 1e-7) < 1e-12
