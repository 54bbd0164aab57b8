"""Test configuration: the ``gpu`` marker and shared helpers.

Tests marked ``gpu`` need a CUDA device and the compiled library; everything
else runs on the CPU (oracle pins, host logic, library symbol checks).
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the compiled CUDA library")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_sessionfinish(session, exitstatus):
    """Write every attention comparison of the run (error and reference
    magnitudes) to the JSON file named by PA_PARITY_LOG, if set."""
    path = os.environ.get("PA_PARITY_LOG")
    if not path:
        return
    mod = sys.modules.get("gpu_util")
    if mod is None:
        return
    import json
    rows = [{"what": w, "max_err": a, "mean_err": b, "max_ref": c, "mean_ref": d,
             "max_ratio": (a / c) if c > 0 else None, "mean_ratio": (b / d) if d > 0 else None}
            for (w, a, b, c, d) in mod.PARITY_LOG]
    with open(path, "w") as f:
        json.dump(rows, f, indent=1)
