"""Closed forms of the speed-up analysis (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

* Expected tokens per target pass, E = (1 - a^(K+1)) / (1 - a)
  ("期望加速比" of "投机解码与 EAGLE"; section 二 of "064 · 投机解码").
* Expected speed-up S = E / (1 + K c) (section 二 of "064 · 投机解码").
* Target work per emitted token relative to plain decoding, when a verify pass
  over K+1 positions costs K+1 single-position passes and the draft is free:
  (K + 1) / E.  "064 · 投机解码" evidence 4 quotes its value at a = 0.8, K = 5.
"""

from __future__ import annotations


def expected_tokens(alpha: float, K: int) -> float:
    if alpha == 1:
        return float(K + 1)
    return (1 - alpha ** (K + 1)) / (1 - alpha)


def speedup(alpha: float, K: int, c: float) -> float:
    return expected_tokens(alpha, K) / (1 + K * c)


def work_ratio(alpha: float, K: int) -> float:
    return (K + 1) / expected_tokens(alpha, K)
