import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_collection_modifyitems(config, items):
    """Tests marked gpu are skipped, not failed, on a host without a GPU."""
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """With MOK_PARITY_REPORT set: the largest |gpu - oracle| / tolerance of
    every named float check that ran, printed and written as JSON to the
    path the variable names."""
    path = os.environ.get("MOK_PARITY_REPORT")
    if not path:
        return
    import json
    from helpers import PARITY_RATIOS
    terminalreporter.write_line("parity: max |gpu - oracle| / tolerance per check")
    for k in sorted(PARITY_RATIOS):
        v = PARITY_RATIOS[k]
        terminalreporter.write_line(f"  {k:64s} {v:.4f}" if isinstance(v, float) else f"  {k:64s} {v}")
    with open(path, "w") as f:
        json.dump(PARITY_RATIOS, f, indent=1, sort_keys=True)
