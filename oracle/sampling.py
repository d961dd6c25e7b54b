"""Per-row building blocks of verification (oracle side, float64).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Every helper that does arithmetic on distributions is written with plain numpy
operations that also work on ``dtype=object`` arrays of ``fractions.Fraction``,
so the exactness tests can run the very same code in exact arithmetic.

Readings taken where the pages are silent:

* Transform order is temperature -> top-k -> top-p, renormalising after each
  truncation; top-k ties go to the lower token index; top-p keeps the shortest
  prefix (probability descending, index ascending) whose cumulative mass
  reaches top_p, always at least one token.  The Leviathan analysis page
  ("064 · 投机解码", section 二) only says p and q must include the temperature
  and top-k / nucleus transform, the same for both.
* Accept test is ``u < p(x)/q(x)`` with u in [0, 1) (exactness rule of
  "投机解码与 EAGLE"; "Bước 1" of the EAGLE-3 lesson); q(x) = 0 accepts
  ("Bước 1": a zero draft probability accepts).
* Residual with zero mass falls back to the target distribution ("Bước 2" of
  the EAGLE-3 lesson returns the verifier distribution when the sum is 0).
* Inverse CDF: the smallest index y with cumsum_{x<=y} w(x) > u * sum(w), in
  vocabulary order.  Zero-weight tokens are never chosen.
"""

from __future__ import annotations

import numpy as np

# Width of the band around a decision threshold inside which a float32 kernel
# and this float64 oracle may legitimately disagree ("near tie").
NEAR_TIE = 1e-5


def _transform_z(z: np.ndarray, top_k: int, top_p: float):
    """z already divided by the temperature.  Returns (probabilities, near_tie)."""
    V = z.size
    idx = np.arange(V)
    order = np.lexsort((idx, -z))  # z descending, index ascending
    keep = order if (top_k <= 0 or top_k >= V) else order[:top_k]
    zk = z[keep]
    m = zk[0]
    if not np.isfinite(m):
        raise ValueError("row has no finite logit")
    e = np.exp(zk - m)
    pk = e / e.sum()
    near = False
    if top_p < 1.0:
        c = np.cumsum(pk)
        hit = np.nonzero(c >= top_p)[0]
        n = int(hit[0]) + 1 if hit.size else keep.size
        near = bool(abs(c[n - 1] - top_p) < NEAR_TIE
                    or (n >= 2 and abs(top_p - c[n - 2]) < NEAR_TIE))
        keep = keep[:n]
        pk = pk[:n] / pk[:n].sum()
    p = np.zeros(V, dtype=np.float64)
    p[keep] = pk
    return p, near


def transform_logits(logits, temperature: float, top_k: int = 0,
                     top_p: float = 1.0):
    """Sampling distribution of one row of logits (temperature > 0)."""
    z = np.asarray(logits, dtype=np.float64) / float(temperature)
    return _transform_z(z, int(top_k), float(top_p))


def transform_probs(probs, temperature: float, top_k: int = 0,
                    top_p: float = 1.0):
    """Same transform for a row given as probabilities: z = log(q) / T."""
    q = np.asarray(probs, dtype=np.float64)
    with np.errstate(divide="ignore"):
        lq = np.where(q > 0, np.log(np.where(q > 0, q, 1.0)), -np.inf)
    return _transform_z(lq / float(temperature), int(top_k), float(top_p))


def transform(row, kind: str, temperature: float, top_k: int = 0,
              top_p: float = 1.0):
    if kind == "logits":
        return transform_logits(row, temperature, top_k, top_p)
    if kind == "probs":
        return transform_probs(row, temperature, top_k, top_p)
    raise ValueError(kind)


def acceptance_mass(p, q):
    """alpha = sum_x min(p(x), q(x)) (acceptance-rate section of the
    Leviathan analysis page)."""
    return np.minimum(p, q).sum()


def accept_prob(p, q, x: int):
    """a(x) = min(1, p(x)/q(x)); q(x) = 0 counts as 1."""
    if q[x] == 0:
        return 1
    r = p[x] / q[x]
    return r if r < 1 else 1


def accept(p, q, x: int, u: float):
    """Returns (accepted, near_tie, q_was_zero) for the draw u."""
    if q[x] == 0:
        return True, False, True
    ratio = p[x] / q[x]
    return bool(u < ratio), bool(abs(u - ratio) < NEAR_TIE), False


def residual(p, q):
    """norm(max(0, p - q)); returns (distribution, used_fallback).

    EAGLE-2 notes §2.1 and the Leviathan page's r(x); zero mass -> p."""
    r = np.maximum(p - q, 0)
    z = r.sum()
    if z == 0:
        return p, True
    return r / z, False


def without_token(q, x: int):
    """Draft distribution after its token x was drawn and rejected: x removed,
    the rest renormalised.  Returns None when no mass is left."""
    q2 = q.copy()
    q2[x] = 0
    s = q2.sum()
    if s == 0:
        return None
    return q2 / s


def inverse_cdf(w, u: float):
    """Smallest y with cumsum(w)[y] > u * sum(w).  Returns (y, near_tie)."""
    c = np.cumsum(np.asarray(w, dtype=np.float64))
    total = c[-1]
    t = u * total
    y = int(np.searchsorted(c, t, side="right"))
    if y >= c.size:  # rounding left no crossing: last positive weight
        y = int(np.nonzero(np.asarray(w) > 0)[0][-1])
    lo = c[y - 1] if y > 0 else 0.0
    near = bool((t - lo) < NEAR_TIE * total or (c[y] - t) < NEAR_TIE * total)
    return y, near


def argmax_first(row):
    """Greedy rule target ("贪婪情形简化" of "投机解码与 EAGLE"): index of the
    largest logit, ties to the lowest index.  NaN is read as -inf, so an
    all-NaN row gives 0."""
    x = np.asarray(row, dtype=np.float64)
    return int(np.argmax(np.where(np.isnan(x), -np.inf, x)))
