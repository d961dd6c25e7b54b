"""Pins of the oracle's per-row building blocks against what the pages fix.

Each test checks the oracle against something other than itself: values the
pages print (tests/golden/), closed forms, exact rational arithmetic, or an
independent brute force.
"""

import math
import os
from fractions import Fraction as F

import numpy as np
import pytest

from oracle import analysis, philox
from oracle.sampling import (accept_prob, acceptance_mass, argmax_first,
                             inverse_cdf, residual, transform_logits,
                             transform_probs)


def _frac(s):
    return None if s == "-" else F(s)


def _load_two_token(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "leviathan_two_token.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line.split())
    return rows


def _exact_output(p, q):
    """Output law of one accept/reject step using the oracle's helpers:
    draft x ~ q, accept with a(x), else draw from the residual."""
    acc = [q[x] * accept_prob(p, q, x) for x in range(len(p))]
    rej = 1 - sum(acc)
    r, _ = residual(p, q)
    return [acc[x] + rej * r[x] for x in range(len(p))]


def test_two_token_examples(golden_dir):
    rows = _load_two_token(golden_dir)
    assert len(rows) == 2
    for name, pa, pb, qa, qb, aa, ab, alpha, fa, fb, wa, wb in rows:
        p = np.array([F(pa), F(pb)], dtype=object)
        q = np.array([F(qa), F(qb)], dtype=object)
        if _frac(aa) is not None:
            assert accept_prob(p, q, 0) == F(aa), name
        assert accept_prob(p, q, 1) == F(ab), name
        assert acceptance_mass(p, q) == F(alpha), name
        out = _exact_output(p, q)
        assert out == [F(fa), F(fb)], name
        # the wrong rule of the page: resample from p on rejection
        acc = [q[x] * accept_prob(p, q, x) for x in range(2)]
        rej = 1 - sum(acc)
        wrong = [acc[x] + rej * p[x] for x in range(2)]
        if _frac(wa) is not None:
            assert wrong[0] == F(wa), name
        assert wrong[1] == F(wb), name


@pytest.mark.parametrize("V", [2, 3, 4])
def test_exact_lossless_random_rationals(V):
    rng = np.random.default_rng(7 + V)
    for _ in range(200):
        a = rng.integers(0, 6, V)
        c = rng.integers(0, 6, V)
        if a.sum() == 0 or c.sum() == 0:
            continue
        p = np.array([F(int(x), int(a.sum())) for x in a], dtype=object)
        q = np.array([F(int(x), int(c.sum())) for x in c], dtype=object)
        assert _exact_output(p, q) == list(p)


def test_alpha_is_one_minus_tv():
    rng = np.random.default_rng(3)
    for V in (2, 17, 1000):
        for _ in range(20):
            p, _ = transform_logits(rng.normal(0, 2, V), 1.0)
            q, _ = transform_logits(rng.normal(0, 2, V), 0.7)
            tv = 0.5 * np.abs(p - q).sum()
            assert abs(acceptance_mass(p, q) - (1 - tv)) < 1e-12


def test_residual_zero_mass_falls_back_to_p():
    p = np.array([0.25, 0.75])
    r, fb = residual(p, p.copy())
    assert fb and r is p


def _closed_forms(golden_dir):
    out = []
    with open(os.path.join(golden_dir, "closed_forms.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append(line.split())
    return out


def test_closed_form_values(golden_dir):
    rows = _closed_forms(golden_dir)
    assert len(rows) == 7
    for fn, *args in rows:
        vals = [float(x) for x in args]
        want, tol = vals[-2], vals[-1]
        if fn == "expected_tokens":
            got = analysis.expected_tokens(vals[0], int(vals[1]))
        elif fn == "speedup":
            got = analysis.speedup(vals[0], int(vals[1]), vals[2])
        else:
            got = analysis.work_ratio(vals[0], int(vals[1]))
        assert abs(got - want) <= tol + 1e-12, (fn, args, got)


def test_expected_tokens_is_geometric_series():
    # E = 1 + a + ... + a^K (section 二 of "064 · 投机解码")
    for a in (0.1, 0.5, 0.8, 0.95):
        for K in range(0, 9):
            assert abs(analysis.expected_tokens(a, K)
                       - sum(a ** i for i in range(K + 1))) < 1e-12


# ---------------------------------------------------------------- transform

def _brute_topk_topp(z, k, top_p):
    """Independent brute force: Python tuple sort, explicit loops."""
    V = len(z)
    ranked = sorted(range(V), key=lambda i: (-z[i], i))
    kept = ranked if (k <= 0 or k >= V) else ranked[:k]
    m = max(z[i] for i in kept)
    w = {i: math.exp(z[i] - m) for i in kept}
    s = sum(w.values())
    pr = {i: w[i] / s for i in kept}
    if top_p < 1:
        acc, keep2 = 0.0, []
        for i in kept:  # already probability-descending, index-ascending
            keep2.append(i)
            acc += pr[i]
            if acc >= top_p:
                break
        s2 = sum(pr[i] for i in keep2)
        pr = {i: pr[i] / s2 for i in keep2}
    out = np.zeros(V)
    for i, v in pr.items():
        out[i] = v
    return out


@pytest.mark.parametrize("V", [1, 5, 16, 64])
def test_transform_matches_brute_force(V):
    rng = np.random.default_rng(V)
    for trial in range(40):
        # integers make exact ties likely
        z = rng.integers(-3, 4, V).astype(np.float64)
        k = int(rng.integers(0, V + 2))
        top_p = float(rng.choice([1.0, 0.9, 0.5, 0.2]))
        T = float(rng.choice([1.0, 0.7, 2.0]))
        got, _ = transform_logits(z, T, k, top_p)
        want = _brute_topk_topp(list(z / T), k, top_p)
        assert np.array_equal(got > 0, want > 0), (trial, k, top_p)
        assert np.allclose(got, want, rtol=1e-12, atol=0)


def test_transform_probs_is_power_and_renormalise():
    rng = np.random.default_rng(11)
    q = rng.dirichlet(np.ones(50))
    q[3] = 0.0
    q = q / q.sum()
    for T in (1.0, 0.5, 1.7):
        got, _ = transform_probs(q, T)
        want = q ** (1 / T)
        want /= want.sum()
        assert np.allclose(got, want, rtol=1e-12, atol=1e-300)
        assert got[3] == 0


def test_greedy_argmax_reduces_to_numpy():
    rng = np.random.default_rng(5)
    for _ in range(200):
        x = rng.integers(-2, 3, 37).astype(np.float32)
        assert argmax_first(x) == int(np.argmax(x))
    assert argmax_first(np.array([np.nan, 1.0, 1.0])) == 1
    assert argmax_first(np.array([np.nan, np.nan])) == 0
    assert argmax_first(np.array([-np.inf, -np.inf, 0.0])) == 2


def test_inverse_cdf_brute_force():
    rng = np.random.default_rng(9)
    for _ in range(300):
        w = rng.random(9) * (rng.random(9) < 0.6)
        if w.sum() == 0:
            continue
        u = float(rng.random())
        y, _ = inverse_cdf(w, u)
        # brute force: walk until the running sum exceeds u * total
        t, acc, want = u * w.sum(), 0.0, None
        for i, x in enumerate(w):
            acc += x
            if acc > t:
                want = i
                break
        assert y == want
        assert w[y] > 0


def test_inverse_cdf_frequencies():
    w = np.array([0.1, 0.0, 0.5, 0.4])
    us = (np.arange(100000) + 0.5) / 100000
    ys = np.array([inverse_cdf(w, float(u))[0] for u in us[::10]])
    freq = np.bincount(ys, minlength=4) / ys.size
    assert np.allclose(freq, w, atol=1e-3)


# ------------------------------------------------------------------- Philox

def test_philox_uniform_range_and_resolution():
    us = philox.uniform_np(1234, np.arange(1 << 16), 3, 0)
    assert us.min() >= 0 and us.max() < 1
    assert np.all((us * (1 << 24)) == np.floor(us * (1 << 24)))


def test_philox_scalar_equals_vectorised():
    rng = np.random.default_rng(0)
    for _ in range(50):
        c = [int(x) for x in rng.integers(0, 2**32, 4, dtype=np.uint64)]
        seed = int(rng.integers(0, 2**63))
        w1 = philox.philox4x32_10(c, philox.seed_key(seed))
        w2 = philox.philox4x32_10_np(*[np.uint64(x) for x in c], seed)
        assert tuple(int(x) for x in w2) == w1


def test_philox_uniformity_chi_square():
    # 2^16 draws into 64 bins; chi-square 99.9% critical value for 63 dof is
    # about 103.4
    us = philox.uniform_np(7, 0, np.arange(1 << 16), 1)
    counts = np.bincount((us * 64).astype(int), minlength=64)
    e = us.size / 64
    chi2 = ((counts - e) ** 2 / e).sum()
    assert chi2 < 103.4


def test_philox_round_is_a_bijection_on_small_domain():
    # With the key fixed, distinct counters give distinct outputs (the map is
    # a bijection); spot-check 2^16 counters that differ in every word.
    ctr = np.arange(1 << 16, dtype=np.uint64)
    w = philox.philox4x32_10_np(ctr, ctr * np.uint64(3), ctr ^ np.uint64(5),
                                np.uint64(9), 42)
    packed = set(zip(*(x.tolist() for x in w)))
    assert len(packed) == 1 << 16


def test_philox_round_matches_multiword_product():
    # One round must equal the high/low halves of the 64-bit products.
    rng = np.random.default_rng(1)
    for _ in range(100):
        c = [int(x) for x in rng.integers(0, 2**32, 4, dtype=np.uint64)]
        k = [int(x) for x in rng.integers(0, 2**32, 2, dtype=np.uint64)]
        out = philox.philox_round(c, k)
        prod0 = divmod(philox.M0 * c[0], 2**32)
        prod1 = divmod(philox.M1 * c[2], 2**32)
        assert out == (prod1[0] ^ c[1] ^ k[0], prod1[1],
                       prod0[0] ^ c[3] ^ k[1], prod0[1])


def _exact_inverse_cdf(w, u):
    """Smallest y with sum_{x<=y} w(x) > u * sum(w), in exact arithmetic:
    float64 weights are scaled to integers by a common power of two, and u
    is a 24-bit dyadic (k / 2^24), so every comparison is between integers."""
    import math
    w = np.asarray(w, dtype=np.float64)
    fr = [math.frexp(float(x)) for x in w]          # x = m * 2^e, 0.5<=m<1
    emin = min(e for m, e in fr if m != 0.0) - 53
    ints = [int(m * (1 << 53)) << (e - 53 - emin) if m != 0.0 else 0
            for m, e in fr]
    total = sum(ints)
    k = int(round(u * (1 << 24)))
    assert k / (1 << 24) == u
    acc = 0
    for y, v in enumerate(ints):
        acc += v
        if (acc << 24) > k * total:
            return y
    return None


@pytest.mark.slow
def test_inverse_cdf_large_vocab_against_exact_arithmetic():
    # residual rows at V = 128256 (the workloads' vocabulary): the oracle's
    # float64 draw equals the exact one wherever it reports no near tie (the
    # 1e-5 band is about one token's mass here, so about a third are skipped)
    rng = np.random.default_rng(31)
    V = 128256
    checked = 0
    for row in range(5):
        zt = rng.normal(0, 2.0, V)
        zq = zt + rng.normal(0, 0.8, V)
        p, _ = transform_logits(zt, 1.0)
        q, _ = transform_logits(zq, 1.0)
        r, _ = residual(p, q)
        for u in rng.integers(0, 1 << 24, size=8) / float(1 << 24):
            y, near = inverse_cdf(r, float(u))
            if near:
                continue
            assert y == _exact_inverse_cdf(r, float(u))
            checked += 1
    assert checked >= 15
