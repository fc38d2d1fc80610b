import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload")


@pytest.fixture(scope="session")
def olib():
    import oracle

    return oracle.lib()


@pytest.fixture(scope="session")
def wl():
    import workload

    workload.lib()
    return workload


def pytest_terminal_summary(terminalreporter):
    """Print what the parity checks logged: excluded near-ties and error ratios per case."""
    support = sys.modules.get("support")
    lines = getattr(support, "REPORT", None) if support else None
    if lines:
        terminalreporter.section("parity report")
        for line in lines:
            terminalreporter.write_line(line)
