import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the CUDA library")
    config.addinivalue_line("markers", "slow: long-running check at full workload size")


def pytest_collection_modifyitems(config, items):
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


def pytest_sessionfinish(session, exitstatus):
    """With FA_PARITY_REPORT set, write every recorded comparison (test,
    tensor, relative Frobenius error, un-discounted max-abs, max |ref|) there
    as JSON."""
    path = os.environ.get("FA_PARITY_REPORT")
    if not path:
        return
    try:
        import json

        from harness import RECORDS
    except Exception:  # pragma: no cover
        return
    d = os.path.dirname(os.path.abspath(path))
    os.makedirs(d, exist_ok=True)
    with open(path, "w") as f:
        json.dump(RECORDS, f, indent=0)
