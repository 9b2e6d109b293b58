import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload")


def read_golden(name):
    """Key -> list of tokens, from a golden fixture (lines starting with # are citations)."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            out.setdefault(key, []).append(rest)
    return out


@pytest.fixture(scope="session")
def golden():
    return read_golden


# Near-tie decisions: discrete outputs whose oracle margin is below the float
# tolerance may legitimately differ from the oracle's; the parity tests count
# them instead of failing, and the counts are reported at the end of the run.
_NEAR_TIES = []


@pytest.fixture
def near_ties(request):
    """Call with the number of near-tie decisions a test met (it is reported, not failed)."""
    def record(n: int) -> int:
        _NEAR_TIES.append((request.node.nodeid, int(n)))
        return int(n)
    return record


def pytest_terminal_summary(terminalreporter):
    if not _NEAR_TIES:
        return
    terminalreporter.section("near-tie decisions (oracle margin below the tolerance: counted, not failed)")
    for nodeid, n in _NEAR_TIES:
        terminalreporter.write_line(f"{n:4d}  {nodeid}")
    terminalreporter.write_line(f"total {sum(n for _, n in _NEAR_TIES)} near-tie decisions in {len(_NEAR_TIES)} tests")
