import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: large CPU oracle work")


def pytest_terminal_summary(terminalreporter):
    """Report, next to the pass/fail bar, how many outputs of each tolerance check are a
    BF16 neighbour of the fp64 reference (the tighter 'within one BF16 ulp' figure) and the
    largest error as a fraction of the bar."""
    try:
        from helpers import FAITHFUL_REPORT
    except ImportError:
        return
    if not FAITHFUL_REPORT:
        return
    tr = terminalreporter
    tr.section("BF16 faithful-rounding report (fraction within one BF16 ulp of the fp64 reference)")
    for what, frac, size, worst in FAITHFUL_REPORT:
        tr.write_line("%-48s %9d outputs  within 1 ulp: %.5f  max err / bar: %.3f" % (what[:48], size, frac, worst))
