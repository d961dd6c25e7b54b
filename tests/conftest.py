import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long Monte-Carlo pin")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


def pytest_terminal_summary(terminalreporter):
    """Near-tie report of the GPU parity tests: per comparison, sequences
    compared element by element, excluded as near ties, and final draws that
    needed the CDF band."""
    mod = sys.modules.get("tests._parity")
    rep = getattr(mod, "REPORT", None)
    if not rep:
        return
    tr = terminalreporter
    tr.section("parity: near ties counted and reported")
    tot = [0, 0, 0, 0]
    for p in rep:
        tr.write_line(f"{p.test}: sequences {p.sequences}, compared "
                      f"{p.compared} (exact {p.exact}, cdf band {p.cdf_band}), "
                      f"near-tie excluded {p.near_tie_excluded}")
        for k, v in enumerate((p.sequences, p.compared, p.near_tie_excluded,
                               p.cdf_band)):
            tot[k] += v
    tr.write_line(f"total: sequences {tot[0]}, compared {tot[1]}, near-tie "
                  f"excluded {tot[2]}, cdf band {tot[3]}")
    out = os.environ.get("SPEC_PARITY_REPORT")
    if out:
        import json
        with open(out, "w") as f:
            json.dump([p.as_dict() for p in rep], f, indent=1)
