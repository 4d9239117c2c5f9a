import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libspc.so")
    config.addinivalue_line("markers", "slow: long-running")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA GPU on this machine")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    from tests import swap_log
    if not swap_log.COUNTS:
        return
    terminalreporter.write_sep("-", "tie-band swaps (GPU vs oracle selections; allowed within 2e-3 of the K-th score)")
    for tid, (sw, checked, heads) in sorted(swap_log.COUNTS.items()):
        terminalreporter.write_line(f"{tid}: {sw} swapped positions, {heads} of {checked} selections with a swap")
