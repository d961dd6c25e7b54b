"""The oracle's Philox4x32-10 against an independent library implementation:
Triton's tl.philox (ten rounds), run as a black box in Triton's CPU
interpreter in a subprocess (outputs only; no code shared).  Keys and
counters cover the extremes and random values."""

import json
import os
import random
import subprocess
import sys

import pytest

from oracle import philox

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_philox_equals_library_philox():
    pytest.importorskip("triton")
    rnd = random.Random(20261202)
    cases = [[0, 0, 0, 0, 0],
             [(1 << 64) - 1, 0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF],
             [1, 0, 3, 1, 0], [1 << 32, 7, 0, 0, 9]]
    cases += [[rnd.getrandbits(64)] + [rnd.getrandbits(32) for _ in range(4)]
              for _ in range(60)]
    r = subprocess.run([sys.executable, os.path.join(HERE, "_triton_philox.py")],
                       input=json.dumps(cases), capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    got = json.loads(r.stdout)
    for c, g in zip(cases, got):
        assert list(philox.philox4x32_10(c[1:], philox.seed_key(c[0]))) == g, c
