"""Pins of the chain verifier: losslessness by Monte-Carlo (the exercises of
"投机解码与 EAGLE" and the EAGLE-3 / Spanish lessons ask for a 1e5-trial KL
check and a 50k-sample chi-square), the expected-token closed form, the greedy
rule, and plain invariants."""

import numpy as np
import pytest
from scipy import stats

from oracle import analysis
from oracle.chain import verify_chain
from oracle.sampling import transform_logits


def _draw(rng, dist, n):
    return rng.choice(dist.size, size=n, p=dist)


def _setup(V, K, seed, noise=0.7, T=1.0):
    rng = np.random.default_rng(seed)
    tl = rng.normal(0, 2.0, (K + 1, V))
    dl = tl[:K] + rng.normal(0, noise, (K, V))
    ps = [transform_logits(tl[k], T)[0] for k in range(K + 1)]
    qs = [transform_logits(dl[k], T)[0] for k in range(K)]
    return rng, tl, dl, ps, qs


def _kl(freq, p):
    m = freq > 0
    return float((freq[m] * np.log(freq[m] / p[m])).sum())


@pytest.mark.parametrize("K", [1, 3])
def test_chain_monte_carlo_lossless(K):
    V, n = 5, 100_000
    rng, tl, dl, ps, qs = _setup(V, K, seed=10 + K)
    toks = np.stack([_draw(rng, qs[k], n) for k in range(K)], axis=1)
    tgt = np.broadcast_to(tl, (n, K + 1, V))
    dft = np.broadcast_to(dl, (n, K, V))
    res = verify_chain(tgt, dft, toks, temperature=1.0, seed=99)
    first = res.tokens[:, 0]
    freq = np.bincount(first, minlength=V) / n
    assert _kl(freq, ps[0]) < 1e-3
    chi2, pval = stats.chisquare(np.bincount(first, minlength=V), ps[0] * n)
    assert pval > 1e-3
    # second token, conditional on the first draft being accepted
    sel = res.accepted >= 1
    sec = res.tokens[sel, 1]
    cnt = np.bincount(sec, minlength=V)
    chi2, pval = stats.chisquare(cnt, ps[1] * cnt.sum())
    assert pval > 1e-3
    # the residual never re-emits the rejected token
    rej = res.accepted == 0
    assert not np.any(res.tokens[rej, 0] == toks[rej, 0])


def test_chain_expected_tokens_closed_form():
    # identical rows at every position -> acceptance is Bernoulli(alpha) at
    # each step, so E[accepted + 1] = (1 - alpha^(K+1)) / (1 - alpha)
    V, K, n = 6, 4, 60_000
    rng = np.random.default_rng(21)
    t = rng.normal(0, 2, V)
    d = t + rng.normal(0, 0.9, V)
    p = transform_logits(t, 1.0)[0]
    q = transform_logits(d, 1.0)[0]
    alpha = np.minimum(p, q).sum()
    toks = _draw(rng, q, n * K).reshape(n, K)
    res = verify_chain(np.broadcast_to(t, (n, K + 1, V)),
                       np.broadcast_to(d, (n, K, V)), toks, temperature=1.0,
                       seed=5)
    emitted = res.accepted.astype(np.float64) + 1
    want = analysis.expected_tokens(alpha, K)
    se = emitted.std() / np.sqrt(n)
    assert abs(emitted.mean() - want) < 5 * se
    assert np.allclose(res.mass, alpha, rtol=1e-12)
    # P(accepted >= k) = alpha^k
    for k in range(1, K + 1):
        frac = (res.accepted >= k).mean()
        assert abs(frac - alpha ** k) < 5 * np.sqrt(alpha ** k / n)


def test_chain_with_topk_topp_is_lossless_for_the_transformed_target():
    V, K, n = 12, 1, 60_000
    rng = np.random.default_rng(4)
    tl = rng.normal(0, 2, (K + 1, V))
    dl = tl[:K] + rng.normal(0, 1, (K, V))
    kw = dict(temperature=0.7, top_k=6, top_p=0.9)
    p0 = transform_logits(tl[0], 0.7, 6, 0.9)[0]
    q0 = transform_logits(dl[0], 0.7, 6, 0.9)[0]
    toks = _draw(rng, q0, n).reshape(n, 1)
    res = verify_chain(np.broadcast_to(tl, (n, K + 1, V)),
                       np.broadcast_to(dl, (n, K, V)), toks, seed=3, **kw)
    cnt = np.bincount(res.tokens[:, 0], minlength=V)
    assert np.all(cnt[p0 == 0] == 0)
    m = p0 > 0
    chi2, pval = stats.chisquare(cnt[m], p0[m] * n)
    assert pval > 1e-3


def test_chain_greedy_brute_force():
    rng = np.random.default_rng(8)
    B, K, V = 50, 5, 9
    tl = rng.integers(-2, 3, (B, K + 1, V)).astype(np.float32)
    g = np.argmax(tl, axis=2)
    toks = np.where(rng.random((B, K)) < 0.7, g[:, :K],
                    rng.integers(0, V, (B, K)))
    res = verify_chain(tl, None, toks, temperature=0.0)
    for b in range(B):
        n = 0
        while n < K and toks[b, n] == g[b, n]:
            n += 1
        assert res.accepted[b] == n
        assert list(res.tokens[b, :n]) == list(toks[b, :n])
        assert res.tokens[b, n] == g[b, n]
        assert np.all(res.tokens[b, n + 1:] == -1)
        assert np.array_equal(res.mass[b], (toks[b] == g[b, :K]).astype(float))


def test_chain_identical_rows_accept_everything():
    rng = np.random.default_rng(2)
    B, K, V = 20, 4, 30
    tl = rng.normal(0, 2, (B, K + 1, V))
    toks = rng.integers(0, V, (B, K))
    res = verify_chain(tl, tl[:, :K].copy(), toks, temperature=1.0, seed=1)
    assert np.all(res.accepted == K)
    assert np.allclose(res.mass, 1.0)


def test_chain_zero_draft_probability_accepts_and_flags():
    V = 4
    t = np.zeros((1, 2, V))
    d = np.array([[[0.0, 0.0, -np.inf, 0.0]]])
    res = verify_chain(t, d, np.array([[2]]), temperature=1.0)
    assert res.accepted[0] == 1 and res.status & 2


def test_chain_out_of_range_token_rejects_and_flags():
    rng = np.random.default_rng(0)
    t = rng.normal(0, 1, (1, 3, 8))
    res = verify_chain(t, t[:, :2], np.array([[1, 99]]), temperature=1.0)
    assert res.accepted[0] == 1 and res.status & 64
