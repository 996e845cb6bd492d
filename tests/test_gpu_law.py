"""GPU parity of the sampling laws and of acceptance from logits ("Module 11.
Speculative Decoding and Quantization", §4: temperature, top-k and top-p
applied to the target and the draft alike before acceptance).

* ``spec_sampling_law`` against the oracle's double-precision law: the kept set
  is identical except where p lies within 1e-5 of a cumulative mass at the cut,
  and every probability within 2e-5 relative (fp32 exp against double); at such
  a cut the kept set must still be a top set whose mass reaches p within 1e-5.
* ``spec_accept_logits`` against ``spec_accept`` on ``spec_sampling_law``'s
  outputs: bit-identical on every row (the same device law function).
* ``spec_accept_logits`` against the oracle's acceptance on the oracle's laws:
  identical on every row whose decisions are not within 1e-5 of a tie (near
  cut, near an acceptance threshold u*q = p, or u within 1e-5 of a bin edge).
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import cuda_or_skip

pytestmark = pytest.mark.gpu

NEAR = 1e-5


def _logits(R, V, seed, std=3.0):
    rng = workloads.host_rng(seed, 40)
    return (rng.standard_normal((R, V), dtype=np.float32) * np.float32(std)).astype(np.float32)


@pytest.fixture
def env():
    return cuda_or_skip()


@pytest.fixture(params=["cluster16", "cluster", "row"])
def form(request, monkeypatch):
    """Every kernel form of the laws: one cluster per row of 8192-logit slices
    (up to 16 CTAs) or of 16384-logit slices (up to 8), or one CTA per row
    streaming the row for each pass (the library picks by row count)."""
    monkeypatch.setenv("MXS_LAW_FORM", request.param)
    return request.param


def _law_gpu(env, l, **kw):
    torch, mxs = env
    dev = torch.device("cuda:0")
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = mxs.spec_sampling_law(torch.from_numpy(l).to(dev), dev_status=status, **kw)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(status.item())


def _check_law(got, l, temperature=1.0, top_k=0, top_p=1.0):
    """Rows whose top-p cut is not within 1e-5 of a tie: the same kept set and
    probabilities within 2e-5.  The other rows ("near"): what is kept is a top
    set whose mass under the top-k law reaches p within 1e-5 and would not
    without its least probable tokens (one logit value: ties are kept
    together), and the probabilities are that law
    renormalised over it.  Returns the number of near rows."""
    ref, margin, kept = oracle.sampling_law(l, temperature, top_k, top_p)
    base, _, _ = oracle.sampling_law(l, temperature, top_k, 1.0)
    near = np.atleast_1d(margin < NEAR)
    got2, ref2, base2, l2 = (a.reshape(-1, a.shape[-1]) for a in (got, ref, base, l))
    for r in range(got2.shape[0]):
        keep = got2[r] > 0
        if not near[r]:
            assert np.array_equal(keep, ref2[r] > 0), r
            np.testing.assert_allclose(got2[r], ref2[r], rtol=2e-5, atol=1e-30)
            continue
        drop = ~keep & np.isfinite(l2[r])
        assert not drop.any() or l2[r][keep].min() > l2[r][drop].max(), r
        mass = base2[r][keep].sum()
        lowest = keep & (l2[r] == l2[r][keep].min())  # ties at the cut are kept together
        assert mass >= top_p - NEAR and mass - base2[r][lowest].sum() < top_p + NEAR, r
        np.testing.assert_allclose(got2[r][keep], base2[r][keep] / mass, rtol=2e-5)
    sums = got2.sum(axis=-1)[np.atleast_1d(kept).reshape(-1) > 0]
    assert np.allclose(sums, 1.0, atol=1e-5)
    return int(near.sum())


@pytest.mark.parametrize("V", [1, 7, 1000, 16384, 16385, 50257, 128256, 131072])
def test_law_plain_softmax(env, form, V):
    l = _logits(6, V, seed=V)
    got, st = _law_gpu(env, l)
    assert st == 0
    assert _check_law(got, l) == 0


@pytest.mark.parametrize("temperature,top_k,top_p", [
    (1.0, 50, 1.0), (0.7, 0, 0.9), (1.5, 40, 0.8), (0.3, 1, 1.0), (1.0, 0, 1e-6), (1.0, 128255, 0.999),
    (2.0, 1000, 0.5), (1.0, 3, 0.999999)])
def test_law_filters(env, form, temperature, top_k, top_p):
    V = 128256
    l = _logits(24, V, seed=int(temperature * 10) + top_k)
    got, st = _law_gpu(env, l, temperature=temperature, top_k=top_k, top_p=top_p)
    assert st == 0
    _check_law(got, l, temperature, top_k, top_p)


@pytest.mark.parametrize("std,kw", [(0.01, {"top_p": 0.5}), (0.01, {"top_k": 1000}), (30.0, {"top_p": 0.99}),
                                    (3.0, {"top_k": 60000, "top_p": 0.999999}), (0.3, {"temperature": 0.05, "top_p": 0.9}),
                                    (3.0, {"temperature": 20.0, "top_k": 5000, "top_p": 0.7})])
def test_law_extreme_spreads(env, form, std, kw):
    # flat rows (one fine bin holds thousands of tokens: the radix finish),
    # very peaked rows, and cuts deep in the tail
    l = _logits(8, 128256, seed=int(std * 100) + len(kw), std=std)
    got, st = _law_gpu(env, l, **kw)
    assert st == 0
    _check_law(got, l, kw.get("temperature", 1.0), kw.get("top_k", 0), kw.get("top_p", 1.0))


def test_law_ties_masked_and_rows_without_law(env, form):
    V = 4096
    l = _logits(5, V, seed=3)
    l[0, ::3] = -np.inf                     # masked tokens
    l[1, :200] = l[1].max() + 1.0           # 200 tied at the top: top-k keeps them all
    l[2, 5] = np.nan                        # no law
    l[3, :] = -np.inf                       # no law
    l[4, 9] = np.inf                        # no law
    torch, mxs = env
    got, st = _law_gpu(env, l, top_k=10, top_p=0.95)
    assert st & mxs.DEV_FLAGS["NO_LAW"]
    assert np.all(got[0, ::3] == 0.0)
    assert np.count_nonzero(got[1]) == 200 and np.allclose(got[1, :200], 1 / 200, rtol=1e-6)
    assert np.all(got[2:] == 0.0)
    _check_law(got[:2], l[:2], 1.0, 10, 0.95)


def test_law_deterministic(env, form):
    l = _logits(16, 128256, seed=9)
    a, _ = _law_gpu(env, l, temperature=0.8, top_k=500, top_p=0.9)
    b, _ = _law_gpu(env, l, temperature=0.8, top_k=500, top_p=0.9)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("V,kw", [
    (1, {}), (7, {"top_k": 3}), (1001, {"top_p": 0.9}), (16385, {"temperature": 0.7, "top_k": 50, "top_p": 0.9}),
    (50257, {"top_p": 0.95}), (128256, {"temperature": 0.8, "top_p": 0.9}), (131071, {"top_k": 1000}),
    (128255, {"top_k": 60000, "top_p": 0.999999}), (4099, {"temperature": 0.05, "top_p": 0.5})])
def test_law_forms_bit_identical(env, monkeypatch, V, kw):
    """The kernel forms take the same decisions on the same fixed-point
    weights: every probability is the same bits.  Odd V puts the rows at
    every 4-byte phase, and the second input starts 4 bytes past a 16-byte
    boundary (unaligned heads and tails; probabilities then written with
    another phase than their logits)."""
    torch, mxs = env
    dev = torch.device("cuda:0")
    R = 9
    l = _logits(R, V, seed=V + 5)
    if V > 8:
        l[3] *= np.float32(0.001)   # flat row: thousands of tokens in one fine bin
        l[5, V // 2] = np.nan       # no law
        l[6, : V // 3] = -np.inf    # masked tokens
        l[7, :5] = l[7].max() + 1   # ties at the top
    flat = torch.from_numpy(np.concatenate([np.zeros(1, np.float32), l.ravel()])).to(dev)
    outs = []
    for f in ("cluster16", "cluster", "row"):
        monkeypatch.setenv("MXS_LAW_FORM", f)
        for t in (torch.from_numpy(l).to(dev), flat[1:].view(R, V)):
            outs.append(mxs.spec_sampling_law(t, **kw).cpu().numpy().view(np.uint32))
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert np.array_equal(outs[0], o)
    if V > 8:
        assert not outs[0][5].any() and outs[0][0].any()


def _spec_logits(B, K, V, seed):
    """Target logits N(0, 3), draft logits = target + N(0, 0.4) at the draft
    positions, drafts drawn from the draft's softmax, u ~ U[0, 1)."""
    rng = workloads.host_rng(seed, 41)
    tl = (rng.standard_normal((B, K + 1, V), dtype=np.float32) * np.float32(3.0)).astype(np.float32)
    dl = (tl[:, :K] + rng.standard_normal((B, K, V), dtype=np.float32) * np.float32(0.4)).astype(np.float32)
    u = rng.random((B, K + 1), dtype=np.float32)
    return tl, dl, u


def _drafts(dl_laws, rng):
    B, K, V = dl_laws.shape
    d = np.empty((B, K), np.int32)
    for b in range(B):
        for i in range(K):
            c = np.cumsum(dl_laws[b, i])
            d[b, i] = min(int(np.searchsorted(c, rng.random() * c[-1], side="right")), V - 1)
    return d


@pytest.mark.parametrize("B,K,kw", [(1, 4, {}), (4, 4, {"temperature": 0.7, "top_p": 0.9}),
                                    (16, 4, {"top_k": 50, "top_p": 0.95}), (64, 4, {"temperature": 1.3}),
                                    (64, 7, {"top_k": 200}), (64, 1, {"top_p": 0.8}), (3, 0, {"top_p": 0.9})])
def test_accept_logits_equals_accept_on_written_laws(env, form, B, K, kw):
    torch, mxs = env
    dev = torch.device("cuda:0")
    V = 128256
    tl, dl, u = _spec_logits(B, K, V, seed=B * 10 + K)
    rng = workloads.host_rng(B + K, 42)
    ql_host, _, _ = oracle.sampling_law(dl, kw.get("temperature", 1.0), kw.get("top_k", 0), kw.get("top_p", 1.0)) \
        if K else (np.zeros((B, 0, V)), None, None)
    d = _drafts(ql_host, rng) if K else np.zeros((B, 0), np.int32)
    t_tl, t_dl = torch.from_numpy(tl).to(dev), torch.from_numpy(dl).to(dev)
    t_d, t_u = torch.from_numpy(d).to(dev), torch.from_numpy(u).to(dev)
    flags_a = torch.zeros(B, dtype=torch.int32, device=dev)
    flags_b = torch.zeros(B, dtype=torch.int32, device=dev)
    tok_a, n_a = mxs.spec_accept_logits(t_tl, t_dl, t_d, t_u, row_flags=flags_a, **kw)
    p = mxs.spec_sampling_law(t_tl, **kw)
    q = mxs.spec_sampling_law(t_dl, **kw) if K else torch.empty((B, 0, V), device=dev)
    tok_b, n_b = mxs.spec_accept(p, q, t_d, t_u, row_flags=flags_b)
    torch.cuda.synchronize()
    assert torch.equal(tok_a, tok_b) and torch.equal(n_a, n_b) and torch.equal(flags_a, flags_b)
    if K:
        assert 0 < float(n_a.float().mean()) <= K + 1


@pytest.mark.parametrize("B,K,kw", [(8, 4, {}), (8, 4, {"temperature": 0.8, "top_k": 100, "top_p": 0.9}),
                                    (6, 7, {"top_p": 0.5})])
def test_accept_logits_matches_oracle(env, form, B, K, kw):
    torch, mxs = env
    dev = torch.device("cuda:0")
    V = 128256
    T, k, pp = kw.get("temperature", 1.0), kw.get("top_k", 0), kw.get("top_p", 1.0)
    tl, dl, u = _spec_logits(B, K, V, seed=77 + K)
    pl, pm, _ = oracle.sampling_law(tl, T, k, pp)
    ql, qm, _ = oracle.sampling_law(dl, T, k, pp)
    d = _drafts(ql, workloads.host_rng(5, 43))
    tok_o, n_o, _, edge = oracle.spec_accept(pl, ql, d, u.astype(np.float64), f64=True)
    tok_g, n_g = mxs.spec_accept_logits(torch.from_numpy(tl).to(dev), torch.from_numpy(dl).to(dev),
                                        torch.from_numpy(d).to(dev), torch.from_numpy(u).to(dev), **kw)
    torch.cuda.synchronize()
    tok_g, n_g = tok_g.cpu().numpy(), n_g.cpu().numpy()
    exempt = 0
    for b in range(B):
        j = int(n_o[b]) - 1
        near = edge[b] < NEAR or pm[b, min(j, K)] < NEAR or (j < K and qm[b, j] < NEAR)
        for i in range(min(j + 1, K)):
            pi, qi = pl[b, i, d[b, i]], ql[b, i, d[b, i]]
            near |= abs(u[b, i] * qi - pi) <= NEAR * max(pi, u[b, i] * qi)
        if near:
            exempt += 1
            continue
        assert n_g[b] == n_o[b] and np.array_equal(tok_g[b], tok_o[b]), b
    # a top-p cut among tokens of ~1e-6 mass is within 1e-5 of a tie on most rows;
    # these configurations leave most rows checkable
    assert exempt < B
