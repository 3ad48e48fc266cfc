import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300) and the built extension")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_collection_modifyitems(config, items):
    # GPU tests need a device; on a machine without one they are skipped, not failed.
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """How often a greedy GPU token differed from the oracle's argmax and was
    accepted as a near tie (within the logit tolerance), with the smallest and
    largest oracle margin among those cases."""
    h = sys.modules.get("_harness")
    if h is None or not h.GREEDY_CHECKS[0]:
        return
    esc = h.ESCAPES
    line = f"greedy token checks: {h.GREEDY_CHECKS[0]}, near-tie escapes: {len(esc)}"
    if esc:
        m = [e[0] for e in esc]
        line += f" (oracle margin min {min(m):.2e}, max {max(m):.2e}; first at {esc[0][1]})"
    terminalreporter.write_line(line)
