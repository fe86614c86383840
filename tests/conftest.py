import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_collection_modifyitems(config, items):
    # GPU tests need the device; without one they are skipped, never faked.
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
    """One JSON line per parity check: rows compared with the oracle, rows
    whose oracle key gap at the k / k+1 boundary is below the gap tolerance,
    and rows whose expert ids differed from the oracle's."""
    try:
        from tests.helpers import PARITY_LOG
    except Exception:
        return
    if not PARITY_LOG:
        return
    import json
    tr = terminalreporter
    tr.section("rows differing from the oracle")
    tot = [0, 0, 0]
    for test, rows, near, differ in PARITY_LOG:
        tr.write_line("PARITY " + json.dumps({"test": test, "rows": rows, "near_gap_rows": near,
                                              "differing_rows": differ}))
        tot[0] += rows
        tot[1] += near
        tot[2] += differ
    tr.write_line("PARITY " + json.dumps({"test": "total", "rows": tot[0], "near_gap_rows": tot[1],
                                          "differing_rows": tot[2]}))
