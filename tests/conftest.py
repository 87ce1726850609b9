import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Print the error metrics the GPU parity tests measured (one line per case)."""
    try:
        from gpu_util import REPORT
    except Exception:  # pragma: no cover
        return
    if not REPORT:
        return
    terminalreporter.write_sep("-", "parity metrics (measured)")
    for name in sorted(REPORT):
        vals = ", ".join(f"{k}={v:.4g}" if isinstance(v, float) else f"{k}={v}" for k, v in REPORT[name].items())
        terminalreporter.write_line(f"{name}: {vals}")


def pytest_collection_modifyitems(config, items):
    """Skip GPU tests cleanly on a machine without a GPU when they were not asked for."""
    try:
        import torch

        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    markexpr = config.getoption("-m") or ""
    if "gpu" in markexpr and "not gpu" not in markexpr:
        # Asked for GPU tests explicitly on a machine without one: let them fail loudly.
        return
    skip = pytest.mark.skip(reason="no CUDA GPU on this machine")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)
