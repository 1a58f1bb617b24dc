import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload check")


def pytest_collection_modifyitems(config, items):
    # Without a GPU the gpu-marked tests cannot run; skip rather than fail so
    # that a plain `pytest tests/` on a CPU machine stays green.
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    # the achieved output errors of every parity check of this session
    try:
        from tests.tolerance import ACHIEVED
    except ImportError:  # pragma: no cover
        return
    if not ACHIEVED:
        return
    tr = terminalreporter
    tr.write_sep("-", "achieved output errors (bar: max abs <= max(2e-2, 2^-7 |ref|), rel Frobenius <= 1e-2)")
    for what, err, rel, amax in ACHIEVED:
        tr.write_line(f"{what:48s} max abs {err:.3e}  rel fro {rel:.3e}  max |ref| {amax:.3g}")
