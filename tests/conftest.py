import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Top-k parity totals: rows compared against the oracle, slots that
    differ from its set (each within 1e-3 relative of the k-th score), and
    oracle slots inside that near-tie band."""
    mod = sys.modules.get("_util")
    st = getattr(mod, "TOPK_STATS", None) if mod else None
    if st and st["rows"]:
        terminalreporter.write_line(
            "top-k parity: %d rows compared with the oracle; %d slots differ from its set, all within 1e-3 "
            "relative of the k-th score; %d oracle slots lie in that near-tie band" %
            (st["rows"], st["differ"], st["in_band"]))
