import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_collection_modifyitems(config, items):
    # GPU tests are only meaningful with a device; on a CPU-only host they are
    # reported as skipped when selected explicitly.
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
    try:
        from tolerance import WORST
    except Exception:  # pragma: no cover
        return
    if not WORST:
        return
    tr = terminalreporter
    tr.section("parity: worst |gpu - exact| / tol per output (1.0 = at the bound)")
    tr.write_line(f"{'output':<40} {'worst':>9} {'near-zero only':>15} {'elements':>12}")
    for name in sorted(WORST):
        worst, floor_hits, n = WORST[name]
        tr.write_line(f"{name:<40} {worst:9.4f} {floor_hits:15d} {n:12d}")
