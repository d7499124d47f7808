import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HERE = os.path.dirname(os.path.abspath(__file__))
for p in (ROOT, HERE):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300) and the built library")


@pytest.fixture(scope="session")
def cuda_ok():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a test marked gpu ran without a CUDA device")
    return True


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Print every parity comparison of the session: measured error beside its bound."""
    if "gpu_helpers" not in sys.modules:
        return
    rows = sys.modules["gpu_helpers"].REPORT
    if not rows:
        return
    tr = terminalreporter
    tr.section("parity: measured error vs bound (max|gpu - oracle| / rms(oracle))")
    for test, what, got, bound, note in rows:
        flag = "ok " if got <= bound else "ULP" if "ulps" in note else "BAD"
        tr.write_line(f"{flag} {got:10.3e} <= {bound:8.2e}  {what}  [{test}]{'  ' + note if note else ''}")
