import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size case, minutes of host work")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    # how the kept-set comparisons of this session were decided
    try:
        from tests import harness
    except Exception:
        return
    st = harness.SEL_STATS
    if st["units"]:
        terminalreporter.write_line(
            "selection checks: %d units, %d identical sets, %d differing inside the 1e-5 relative tie "
            "band, %d differing only within the fp32 bound of the pages involved"
            % (st["units"], st["identical"], st["tie_band"], st["fp32_band"]))
