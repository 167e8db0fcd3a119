import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (run with -m gpu)")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Print the flag rates of the GPU-vs-oracle comparisons, when any ran."""
    try:
        from parity_util import FLAG_LOG, flag_report
    except Exception:
        return
    if not FLAG_LOG:
        return
    terminalreporter.write_sep("-", "decision flags (accept band 1e-5; draw band 1e-5/V, "
                                    "literal band 1e-5)")
    for line in flag_report():
        terminalreporter.write_line(line)
