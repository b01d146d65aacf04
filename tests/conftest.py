import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a)")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Reports the INT2 boundary cases (rounding ties excused by the parity
    rule) that the GPU parity tests counted."""
    try:
        from parity_util import BOUNDARY_CASES
    except Exception:
        return
    if not BOUNDARY_CASES:
        return
    tr = terminalreporter
    tr.section("INT2 boundary cases (codes within 1e-6 of a rounding boundary; (s, z) at a rounding tie of their format)")
    tc = ts = tn = 0
    for name, c, z, n in BOUNDARY_CASES:
        tr.write_line("%-40s code ties %4d   (s, z) ties %4d   of %d group records" % (name, c, z, n))
        tc, ts, tn = tc + c, ts + z, tn + n
    tr.write_line("%-40s code ties %4d   (s, z) ties %4d   of %d group records" % ("total", tc, ts, tn))
