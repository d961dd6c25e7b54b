"""Pins of the LM-head oracle (oracle/lmhead.py), none of which uses the
oracle to check itself:

* bf16 rounding equals torch's float32 -> bfloat16 conversion (an
  independent library routine, round-to-nearest-even) on float32 values,
  ties included;
* the bf16 neighbours bracket the value, are bf16 values and are one bf16
  unit apart;
* the exact logits equal brute-force dot products in exact rational
  arithmetic;
* the accumulation-error bound holds for an explicit float32 summation in
  groups of 16, whose bf16 rounding lies in the oracle's [lo, hi] range,
  including sums that cancel to near zero (where the range spans many bf16
  values);
* with logits that are bf16 values already, verification through the LM
  head equals tree verification of those logits, with no rounding ties; an
  accept test whose ratio straddles the uniform under the two roundings is a
  rounding tie.
"""

from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle.lmhead import (bf16_neighbours, bf16_round, lm_head_logits,
                           mass_slack, verify_tree_lmhead)
from oracle.sampling import acceptance_mass, transform
from oracle.tree import verify_tree


def _bf16(a):
    """float64 array of bf16 values (via torch, for inputs only)."""
    return torch.from_numpy(np.asarray(a, np.float32)).bfloat16().double() \
        .numpy()


def test_bf16_round_equals_torch_conversion():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * s
                        for s in (1e-3, 0.5, 3.0, 70.0, 1e5)]).astype(
                            np.float32)
    # exact midpoints between bf16 neighbours: ties go to the even one
    b = _bf16(rng.standard_normal(5000))
    lo, hi = bf16_neighbours(b * (1 + 2.0 ** -7) + 1e-30)
    mids = (0.5 * (lo + hi)).astype(np.float32)
    x = np.concatenate([x, mids, -mids, np.float32([0.5, 1.0, 2.0 ** 20])])
    want = torch.from_numpy(x).bfloat16().double().numpy()
    got = bf16_round(x.astype(np.float64))
    assert np.array_equal(got, want)


def test_bf16_neighbours_bracket_and_are_one_unit_apart():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(50000) * 4.0
    lo, hi = bf16_neighbours(x)
    assert (lo <= x).all() and (x <= hi).all()
    assert np.array_equal(bf16_round(lo), lo)
    assert np.array_equal(bf16_round(hi), hi)
    # one unit in the last of 8 significant bits of the value's binade
    unit = np.ldexp(1.0, np.frexp(np.abs(x))[1] - 8)
    assert np.allclose(hi - lo, unit, rtol=0, atol=0)
    rn = bf16_round(x)
    assert ((rn == lo) | (rn == hi)).all()
    assert (np.abs(rn - x) <= 0.5 * unit).all()
    b = bf16_round(x)  # bf16 values are their own neighbours
    lo, hi = bf16_neighbours(b)
    assert np.array_equal(lo, b) and np.array_equal(hi, b)


def test_exact_logits_equal_rational_dot_products():
    rng = np.random.default_rng(2)
    h = _bf16(rng.standard_normal((3, 24)))
    w = _bf16(rng.standard_normal((7, 24)) * 0.3)
    lg = lm_head_logits(h, w)
    for i in range(3):
        for v in range(7):
            z = sum(Fraction(float(a)) * Fraction(float(c))
                    for a, c in zip(h[i], w[v]))
            assert abs(lg.exact[i, v] - float(z)) <= 1e-14 * max(1, abs(z))
            assert lg.rn[i, v] == bf16_round(float(z))


def test_error_bound_covers_float32_accumulation_in_groups():
    rng = np.random.default_rng(3)
    H, V = 4096, 300
    h = _bf16(rng.standard_normal((4, H)))
    w = _bf16(rng.standard_normal((V, H)) * (2.0 / np.sqrt(H)))
    lg = lm_head_logits(h, w)
    # float32 accumulation: each group of 16 products summed, added to the
    # running float32 sum (products of bf16 values are exact in float32)
    prod = (h[:, None, :] * w[None, :, :]).astype(np.float32)
    acc = np.zeros((4, V), np.float32)
    for g in range(0, H, 16):
        part = np.zeros((4, V), np.float32)
        for t in range(16):
            part = part + prod[:, :, g + t]
        acc = acc + part
    err = np.abs(acc.astype(np.float64) - lg.exact)
    assert (err <= lg.delta).all(), float((err / lg.delta).max())
    # the float32 sum's bf16 rounding lies in the oracle's range, which
    # holds the nearest rounding and is a single value where not ambiguous
    got = bf16_round(acc.astype(np.float64))
    assert ((lg.lo <= got) & (got <= lg.hi)).all()
    assert ((lg.lo <= lg.rn) & (lg.rn <= lg.hi)).all()
    ok = ~lg.ambiguous
    assert np.array_equal(lg.lo[ok], lg.rn[ok])
    assert np.array_equal(lg.hi[ok], lg.rn[ok])
    assert lg.ambiguous.any() and ok.any()
    # away from zero the range is at most the two bf16 neighbours
    big = np.abs(lg.exact) > 1.0
    nlo, nhi = bf16_neighbours(lg.exact[big])
    assert (lg.lo[big] >= nlo).all() and (lg.hi[big] <= nhi).all()


def test_cancelling_sums_span_many_bf16_values():
    # h . w that cancels to about 1e-6: a bf16 unit there is ~1e-14, far
    # below the float32 accumulation error, so the range holds many values
    # and still contains the float32 summation's rounding
    H = 512
    rng = np.random.default_rng(8)
    h = _bf16(rng.standard_normal((1, H)))
    w = _bf16(rng.standard_normal((1, H)) * 0.1)
    w2 = w.copy()
    w2[0, -1] = 0.0  # choose the last product so the sum nearly cancels
    part = float((h @ w2.T)[0, 0])
    w2[0, -1] = _bf16(np.array([-part / h[0, -1]]))[0]
    lg = lm_head_logits(h, w2)
    assert abs(lg.exact[0, 0]) < 1e-2 and lg.ambiguous[0, 0]
    unit = np.ldexp(1.0, np.frexp(abs(lg.rn[0, 0]))[1] - 8)
    assert lg.hi[0, 0] - lg.lo[0, 0] > 4 * unit
    prod = (h * w2).astype(np.float32)[0]
    acc = np.float32(0)
    for g in range(0, H, 16):
        acc = np.float32(acc + prod[g:g + 16].sum(dtype=np.float32))
    got = bf16_round(float(acc))
    assert lg.lo[0, 0] <= got <= lg.hi[0, 0]


def _tree(B=2, V=40, H=8, seed=4):
    rng = np.random.default_rng(seed)
    parent = np.array([[-1, -1, 0, 0, 2]] * B, np.int32)
    N = parent.shape[1]
    toks = np.stack([rng.choice(V, N, replace=False) for _ in range(B)])
    draft = rng.dirichlet(np.ones(V), size=(B, N + 1))
    q_row = np.tile(np.arange(N + 1, dtype=np.int32), (B, 1))
    return parent, toks.astype(np.int32), draft, q_row


def test_lmhead_verification_equals_tree_verification_of_exact_logits():
    # W selects one hidden coordinate per token (one-hot rows), so every
    # logit is a hidden entry: a bf16 value, exact, never ambiguous
    B, V, H = 2, 40, 48
    parent, toks, draft, q_row = _tree(B, V, H)
    rng = np.random.default_rng(5)
    hidden = _bf16(rng.standard_normal((B, parent.shape[1] + 1, H)) * 2)
    w = np.zeros((V, H))
    w[np.arange(V), rng.integers(0, H, V)] = 1.0
    res = verify_tree_lmhead(hidden, w, draft, q_row, toks, parent,
                             temperature=1.0, draft_kind="probs", seed=9)
    z = hidden @ w.T
    want = verify_tree(z, draft, q_row, toks, parent, temperature=1.0,
                       draft_kind="probs", seed=9)
    assert not res.logits.ambiguous.any()
    assert not res.rounding_tie.any()
    assert np.array_equal(res.ref.path_len, want.path_len)
    assert np.array_equal(res.ref.tokens, want.tokens)
    np.testing.assert_array_equal(res.ref.mass, want.mass)


def test_rounding_tie_when_the_two_roundings_decide_differently():
    # one drafted child; its logit sits exactly on a bf16 midpoint, so it is
    # ambiguous, and the uniform lies between the two acceptance ratios
    V, H = 8, 16
    parent = np.array([[-1]], np.int32)
    toks = np.array([[3]], np.int32)
    q = np.full((1, 2, V), 0.6 / (V - 1))
    q[:, :, 3] = 0.4
    q_row = np.array([[0, 1]], np.int32)
    hidden = np.zeros((1, 2, H))
    hidden[0, 0, 0] = 1.0
    w = np.zeros((V, H))
    w[3, 0] = 1.0 + 2.0 ** -8  # midpoint of 1 and 1 + 2^-7
    lg = lm_head_logits(hidden, w)
    assert lg.ambiguous[0, 0, 3] and not lg.ambiguous[0, 0, 2]

    def ratio(z3):
        z = np.zeros(V)
        z[3] = z3
        p = np.exp(z) / np.exp(z).sum()
        return p[3] / q[0, 0, 3]
    r_lo, r_hi = ratio(1.0), ratio(1.0 + 2.0 ** -7)
    u_between = 0.5 * (r_lo + r_hi)
    assert r_lo < u_between < r_hi < 1.0

    def run(u0):
        return verify_tree_lmhead(
            hidden, w, q, q_row, toks, parent, temperature=1.0,
            draft_kind="probs",
            uniform=lambda b, i, slot: u0 if slot == 0 else 0.5)
    assert run(u_between).rounding_tie[0]
    assert run(u_between).ref.near_tie[0]
    assert not run(0.05).rounding_tie[0]    # accepted either way
    assert not run(0.999).rounding_tie[0]   # rejected either way


def test_mass_slack_bounds_any_rounding_in_range():
    # logits taking arbitrary values in [lo, hi] (each ambiguous logit at a
    # random end) move alpha = sum min(p, q) by no more than the slack
    rng = np.random.default_rng(9)
    H, V, T = 512, 3000, 0.8
    h = _bf16(rng.standard_normal((4, H)))
    w = _bf16(rng.standard_normal((V, H)) * (3.0 / np.sqrt(H)))
    lg = lm_head_logits(h, w)
    slack = mass_slack(lg, T)
    assert lg.ambiguous.any() and (slack > 0).all()
    q = rng.dirichlet(np.ones(V) * 0.3, size=4)
    for trial in range(5):
        pick = rng.random(lg.rn.shape) < 0.5
        moved = np.where(lg.ambiguous, np.where(pick, lg.lo, lg.hi), lg.rn)
        for r in range(4):
            p0, _ = transform(lg.rn[r], "logits", T)
            p1, _ = transform(moved[r], "logits", T)
            a0 = acceptance_mass(p0, q[r])
            a1 = acceptance_mass(p1, q[r])
            assert abs(a1 - a0) <= slack[r], (trial, r, a1 - a0, slack[r])
