import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running full-size case")


def pytest_terminal_summary(terminalreporter):
    """Worst max-relative error of every parity case that recorded one, against its limit."""
    mod = sys.modules.get("kda_cases")
    margins = getattr(mod, "MARGINS", None) if mod else None
    if not margins:
        return
    terminalreporter.section("parity margins (max |x - ref| / max |ref|, worst block)")
    for name in sorted(margins):
        err, tol, test, what = margins[name]
        terminalreporter.write_line(f"{name:48s} {err:.3e}   limit {tol:.0e}   ({err / tol:5.1%} of limit)   "
                                    f"worst: {test}, {what}")
