import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter):
    """The worst out / lse errors each parity test measured against the oracle."""
    from tests.parity import STATS
    if not STATS:
        return
    tr = terminalreporter
    tr.section("parity: worst errors against the oracle")
    tr.write_line("%-78s %5s %10s %10s %10s" % ("test", "n", "|dlse|", "rel-L2", "unit-err"))
    for name, s in sorted(STATS.items()):
        tr.write_line("%-78s %5d %10.3e %10.3e %10.3e" % (name[-78:], s["n"], s["lse"], s["rel_l2"],
                                                          s["unit"]))
