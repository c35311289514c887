import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def load_golden(name):
    """Parse a tests/golden/*.txt fixture: '# ...' comment lines, then 'key v1 v2 ...' lines."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = [float(v) for v in vals]
    return out


def pytest_terminal_summary(terminalreporter):
    """Print the near-tie counts the GPU parity tests recorded (rows whose top-K membership, and
    blocks whose walk, the tolerance cannot decide), so that they reach the session's output."""
    try:
        from tests.parity import REPORT
    except Exception:
        return
    if not REPORT:
        return
    terminalreporter.write_line("parity near-tie counts:")
    for name, counts in REPORT:
        terminalreporter.write_line(f"  {name}: " + ", ".join(f"{k}={v}" for k, v in counts.items()))
