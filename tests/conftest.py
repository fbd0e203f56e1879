import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")


def pytest_terminal_summary(terminalreporter):
    from tests.helpers import MARGINS, dump_margins
    if not MARGINS:
        return
    terminalreporter.section("parity margins (achieved error / bar)")
    for name in sorted(MARGINS):
        m = MARGINS[name]
        errs = ", ".join(f"{k} {v:.3g}" for k, v in m.items() if k != "tol")
        worst = max(v for k, v in m.items() if k != "tol")
        terminalreporter.write_line(f"{name}: {errs} (bar {m['tol']:.0e}, worst at {worst / m['tol']:.1%} of it)")
    dump_margins()
